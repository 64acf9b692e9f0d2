"""Plain, slow, double-precision CPU oracle for the int4g path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It
shares no code with the CUDA library (no kernels, headers, tables or helpers);
the two meet only through arrays produced by the seeded input generators.

What it computes, and where it comes from:

* int4g group quantization -- "FastLLM：零依赖CPU推理框架" (pgsm.cn), section
  3.1 "4-bit 量化与权重重排": weights are quantized to 4 bits in groups, commonly
  128 weights per group, each group sharing one scale and one zero point, and
  dequantized to float inside the matmul.  The page gives no formula; the plain
  asymmetric min/max rule is used:
      s = (max - min) / 15,  s16 = fp16(s)  (round to nearest even)
      z = clamp(round(-min / s16), 0, 15)
      q = clamp(round(w / s16) + z, 0, 15)
      w' = s16 * (q - z)
  with round = half away from zero, computed in double.
* the dequantized linear y = x . deq(W)^T  (same section: "read 4-bit weight ->
  dequantize -> matmul" pipeline), and its elementwise error bound
  |y - y_ref| <= 2e-3 * sum_k |x||w'| + 1e-5 on the fp32-accumulated result,
  widened by the final bf16 store (at most 2^-8 of the stored value: bf16 has
  8 significant bits, so that store alone can exceed the first term when
  |y| > 0.51 * sum_k |x||w'|).
* the tile-interleaved weight layout ("按组重排 ... 连续内存", same section):
  an invertible byte/nibble permutation, restated here from its definition.
  Its super-blocks always span 128 columns.  Groups of 256 (same page,
  section 4.2 "模型转换与格式说明": --group-size defaults to 128 and may be
  raised to 256) are stored as two consecutive super-blocks that carry the
  same scale and zero point; the dequantized weights are unchanged.  Groups
  of 64 (section 5.4 "精度与速度平衡": a group size of 64 for more precision)
  keep the super-blocks, which then carry the scale and zero point of the
  first 64 columns, and append a side array with those of the second 64
  columns of every super-block.
* the router projection logits = x . Wr^T in front of the top-k choice (not
  detailed on the pages; the plain dense projection);
* the routed MoE expert FFN with int4g experts -- fastllm README (gittoolsai
  mirror), "2. 如何设定推理精度" (--moe_dtype int4g) and "5. 其它参数"
  (--moe_experts = top-k, --cuda_se = shared expert): top-k routing,
  permutation by expert, SwiGLU gate/up, down projection, gate-weighted
  combine, plus an always-on shared expert with weight 1.

Readings where the pages are silent (tie-breaks, constant groups, storage
order, ...) are stated beside the code that takes them.

Parity pins: every function here is checked by tests/test_oracle_pins.py
against hand-worked cases (tests/golden/), closed forms, invariants and
brute force.  None is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

GROUP = 128          # weights per group along K (FastLLM page, section 3.1)
GROUPS = (64, 128, 256)  # group sizes of the layout (section 4.2: 128 by default, 256 allowed;
                         # section 5.4: 64 for more precision)
SB_SIDE = 320        # groups of 64: per super-block, the second group's 128 scales + 128 zeros
QMAX = 15            # 4-bit codes 0..15
ROW_TILE = 128       # rows per super-block of the interleaved layout
SB_NIB = 8192        # nibble bytes per super-block: 128 rows x 64 B
SB_SCALE = 256       # 128 fp16 scales
SB_ZERO = 64         # 128 4-bit zeros
SB_BYTES = SB_NIB + SB_SCALE + SB_ZERO   # 8512
BF16_U = 2.0 ** -8   # unit roundoff of bf16 (8 significant bits): max relative rounding error


# --------------------------------------------------------------------------
# scalar helpers (exact definitions)
# --------------------------------------------------------------------------

def round_half_away(v):
    """Round to the nearest integer, ties away from zero (C `round`).

    Written as trunc + exact fractional part so that no addition of 0.5 can
    round the argument itself (0.49999999999999994 stays 0).
    """
    v = np.asarray(v, dtype=np.float64)
    t = np.trunc(v)
    frac = v - t                      # exact in binary floating point
    return t + np.where(np.abs(frac) >= 0.5, np.sign(v), 0.0)


def fp16_bits(v):
    """Correctly rounded (nearest even) double -> IEEE half, as uint16 bits.
    Values beyond the half range give infinity (the callers test for it)."""
    with np.errstate(over="ignore"):
        return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


def fp16_value(bits):
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_value(bits):
    """bf16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# --------------------------------------------------------------------------
# a1: quantizer
# --------------------------------------------------------------------------

def quantize_group(w):
    """Quantize one group (1-D array of fp32 values) -> (q[uint8], s16 bits, z).

    Readings where the pages are silent:
      * the scale used for z and q is the stored fp16 s16, so that the
        dequantized weight is exactly what the stored triple encodes;
      * a constant group c: c == 0 -> s16 = 0, z = 0, q = 0; c != 0 -> the
        range [min(c, 0), max(c, 0)] is used, which reconstructs c;
      * s16 == 0 after rounding (range below half the smallest fp16
        subnormal times 15) -> treated as the zero group;
      * s16 overflowing fp16 is an error (ValueError).
    """
    w = np.asarray(w, dtype=np.float32).astype(np.float64)
    n = w.shape[0]
    mn = w.min()
    mx = w.max()
    if mn == mx:
        if mn == 0.0:
            return np.zeros(n, np.uint8), np.uint16(0), 0
        mn, mx = min(mn, 0.0), max(mx, 0.0)
    s = (mx - mn) / QMAX
    sbits = fp16_bits(s)
    s16 = float(fp16_value(sbits))
    if np.isinf(s16) or np.isnan(s16):
        raise ValueError("group scale overflows fp16")
    if s16 == 0.0:
        return np.zeros(n, np.uint8), np.uint16(0), 0
    z = int(np.clip(round_half_away(-mn / s16), 0, QMAX))
    q = np.clip(round_half_away(w / s16) + z, 0, QMAX).astype(np.uint8)
    return q, np.uint16(sbits), z


def quantize(W, group=GROUP):
    """W fp32 [N, K] -> canonical triple (Q, S, Z), by quantize_group applied
    to every group (written with array operations over all groups at once;
    quantize_loops() is the same rule one group at a time, and the pins check
    that the two agree bit for bit).

    Q uint8 [N, K/2]       two codes per byte, low nibble = even k
    S uint16 [N, G]        fp16 scale bits, G = K / group
    Z uint8 [N, ceil(G/2)] two zero points per byte, low nibble = even g
    """
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    if K % group != 0 or K % 2 != 0:
        raise ValueError("K must be a multiple of the group size")
    G = K // group
    w = W.reshape(N, G, group).astype(np.float64)
    mn = w.min(axis=2)
    mx = w.max(axis=2)
    const = mn == mx
    zero = const & (mn == 0.0)
    mn = np.where(const, np.minimum(mn, 0.0), mn)
    mx = np.where(const, np.maximum(mx, 0.0), mx)
    with np.errstate(invalid='ignore', over='ignore', divide='ignore'):
        s = (mx - mn) / QMAX
        sbits = fp16_bits(s)
        s16 = fp16_value(sbits)
        if (~zero & ~np.isfinite(s16)).any():
            raise ValueError("group scale overflows fp16")
        zero = zero | (s16 == 0.0)
        safe = np.where(zero, 1.0, s16)
        z = np.clip(round_half_away(-mn / safe), 0, QMAX)
        q = np.clip(round_half_away(w / safe[:, :, None]) + z[:, :, None], 0, QMAX)
    z = np.where(zero, 0, z).astype(np.uint8)
    q = np.where(zero[:, :, None], 0, q).astype(np.uint8).reshape(N, K)
    S = np.where(zero, 0, sbits).astype(np.uint16)
    return pack_codes(q), S, pack_zeros(z)


def quantize_loops(W, group=GROUP):
    """quantize(), one group at a time through quantize_group."""
    W = np.asarray(W, dtype=np.float32)
    N, K = W.shape
    if K % group != 0 or K % 2 != 0:
        raise ValueError("K must be a multiple of the group size")
    G = K // group
    q = np.zeros((N, K), np.uint8)
    S = np.zeros((N, G), np.uint16)
    z = np.zeros((N, G), np.uint8)
    for n in range(N):
        for g in range(G):
            qq, sb, zz = quantize_group(W[n, g * group:(g + 1) * group])
            q[n, g * group:(g + 1) * group] = qq
            S[n, g] = sb
            z[n, g] = zz
    return pack_codes(q), S, pack_zeros(z)


def pack_codes(q):
    """codes uint8 [N, K] (0..15) -> bytes [N, K/2], low nibble = even k."""
    q = np.asarray(q, np.uint8)
    return (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)


def unpack_codes(Q):
    Q = np.asarray(Q, np.uint8)
    N, Kh = Q.shape
    q = np.empty((N, 2 * Kh), np.uint8)
    q[:, 0::2] = Q & 0xF
    q[:, 1::2] = Q >> 4
    return q


def pack_zeros(z):
    """zero points uint8 [N, G] -> bytes [N, ceil(G/2)], low nibble = even g."""
    z = np.asarray(z, np.uint8)
    N, G = z.shape
    if G % 2:
        z = np.concatenate([z, np.zeros((N, 1), np.uint8)], axis=1)
    return (z[:, 0::2] | (z[:, 1::2] << 4)).astype(np.uint8)


def unpack_zeros(Z, G):
    Z = np.asarray(Z, np.uint8)
    z = np.empty((Z.shape[0], 2 * Z.shape[1]), np.uint8)
    z[:, 0::2] = Z & 0xF
    z[:, 1::2] = Z >> 4
    return z[:, :G]


def dequantize(Q, S, Z, group=GROUP):
    """Canonical triple -> W' float64 [N, K], w' = s16 * (q - z) exactly."""
    q = unpack_codes(Q).astype(np.float64)
    N, K = q.shape
    G = K // group
    s = fp16_value(S).reshape(N, G)
    z = unpack_zeros(Z, G).astype(np.float64)
    qg = q.reshape(N, G, group)
    return (s[:, :, None] * (qg - z[:, :, None])).reshape(N, K)


# --------------------------------------------------------------------------
# a3/a4: dequantized linear and its error bound
# --------------------------------------------------------------------------

def linear(x, Q, S, Z, group=GROUP):
    """y[m, n] = sum_k x[m, k] * w'[n, k] in double.  x: float64 [M, K]."""
    Wd = dequantize(Q, S, Z, group)
    return np.asarray(x, np.float64) @ Wd.T


def _with_output_rounding(bound, y):
    """A bound on the error before the final bf16 store, widened by that store:
    rounding v to bf16 moves it by at most BF16_U*|v| <= BF16_U*(|y| + bound)."""
    return bound * (1.0 + BF16_U) + BF16_U * np.abs(y)


def linear_tolerance(x, Q, S, Z, group=GROUP, rel=2e-3, abs_=1e-5):
    """Elementwise bound rel * sum_k |x[m,k]| |w'[n,k]| + abs_ on the fp32
    result, plus the rounding of the bf16 output (half an ulp, <= 2^-8 |y|)."""
    Wd = dequantize(Q, S, Z, group)
    x = np.asarray(x, np.float64)
    return _with_output_rounding(rel * (np.abs(x) @ np.abs(Wd).T) + abs_, x @ Wd.T)


def linear_columns(x, Q, S, Z, cols, group=GROUP):
    """Only the output columns `cols` of linear() (for sampled checks at full
    size): dequantizes just those weight rows.  Returns (y, tol)."""
    cols = np.asarray(cols)
    Wd = dequantize(Q[cols], S[cols], Z[cols], group)
    x = np.asarray(x, np.float64)
    y = x @ Wd.T
    return y, _with_output_rounding(2e-3 * (np.abs(x) @ np.abs(Wd).T) + 1e-5, y)


# --------------------------------------------------------------------------
# a2: tile-interleaved layout ("int4g-tiled")
# --------------------------------------------------------------------------

def _check_layout(K, group):
    if group not in GROUPS or K % group or K % GROUP:
        raise ValueError("the interleaved layout takes groups of 64, 128 or 256, K % group == 0 and K % 128 == 0")


def tiled_bytes(N, K, group=GROUP):
    """Bytes of the interleaved layout: one 8512-byte super-block per 128
    rows x 128 columns, plus (groups of 64) a 320-byte side entry per
    super-block."""
    _check_layout(K, group)
    Np = -(-N // ROW_TILE) * ROW_TILE
    nsb = (Np // ROW_TILE) * (K // GROUP)
    return nsb * (SB_BYTES + (SB_SIDE if group == 64 else 0))


def expand_groups(S, Z, group):
    """Scales and zero points of a triple with `group` columns per group,
    restated per 128 columns: each group's entry repeated group/128 times
    (the dequantized weights are the same, dequantize() of both agree)."""
    r = group // GROUP
    G = S.shape[1]
    S128 = np.repeat(np.asarray(S, np.uint16), r, axis=1)
    Z128 = pack_zeros(np.repeat(unpack_zeros(Z, G), r, axis=1))
    return S128, Z128


def _nibble_address(kk, r):
    """Position of logical column kk (0..127 inside a group) of row r (0..127
    inside a row tile) in the row's 64 bytes: returns (byte offset, nibble half).

    The 16 32-bit words of a row hold 8 columns each; word slot p holds
    logical word 4*(p%4) + p//4, and inside a word, nibble e holds column
    offset 2*(e%4) + e//4.  Inverted: logical word wl -> p = 4*(wl%4) +
    wl//4, offset o -> e = 4*(o%2) + o//2.  The four 16-byte chunks of row r
    (slots 4c..4c+3 form chunk c) are rotated by (r//2)%4: chunk c sits at
    16-byte position (c + (r//2)%4) % 4.
    """
    kk = np.asarray(kk)
    r = np.asarray(r)
    wl, o = kk // 8, kk % 8
    p = 4 * (wl % 4) + wl // 4
    e = 4 * (o % 2) + o // 2
    pos = (p // 4 + (r // 2) % 4) % 4
    return 16 * pos + 4 * (p % 4) + e // 2, e % 2


def repack(Q, S, Z, N, K, group=GROUP):
    """Canonical triple -> interleaved byte array (uint8, tiled_bytes long).

    Super-block (T, g) -- rows 128T..128T+127, group g -- starts at byte
    (T * G + g) * 8512 and holds: 128 rows x 64 B of codes (row r at r*64,
    columns placed by _nibble_address(kk, r)), then 128 fp16 scales (row r at
    8192 + 2r, little endian), then 128 zero points (row r in byte
    8448 + r//2, low nibble = even r).  Rows past N are zero.

    group 256: the super-blocks still span 128 columns; both super-blocks of
    a group carry that group's scale and zero point (expand_groups).
    """
    _check_layout(K, group)
    if group == 64:
        return _repack_g64(Q, S, Z, N, K)
    if group != GROUP:
        S, Z = expand_groups(S, Z, group)
        group = GROUP
    G = K // group
    Np = -(-N // ROW_TILE) * ROW_TILE
    q = np.zeros((Np, K), np.uint8)
    q[:N] = unpack_codes(Q)
    s = np.zeros((Np, G), np.uint16)
    s[:N] = S
    z = np.zeros((Np, G), np.uint8)
    z[:N] = unpack_zeros(Z, G)
    out = np.zeros(tiled_bytes(N, K, group), np.uint8)
    rows = np.arange(ROW_TILE)
    boff, half = _nibble_address(np.arange(GROUP)[None, :], rows[:, None])   # [128 rows, 128 columns]
    for T in range(Np // ROW_TILE):
        for g in range(G):
            base = (T * G + g) * SB_BYTES
            blk = q[T * ROW_TILE:(T + 1) * ROW_TILE, g * group:(g + 1) * group]
            nib = np.zeros((ROW_TILE, 64), np.uint8)
            for kk in range(GROUP):
                nib[rows, boff[:, kk]] |= (blk[:, kk] << (4 * half[:, kk])).astype(np.uint8)
            out[base:base + SB_NIB] = nib.reshape(-1)
            sc = s[T * ROW_TILE:(T + 1) * ROW_TILE, g]
            out[base + SB_NIB:base + SB_NIB + SB_SCALE] = sc.astype('<u2').view(np.uint8)
            zz = z[T * ROW_TILE:(T + 1) * ROW_TILE, g]
            zb = np.zeros(SB_ZERO, np.uint8)
            for r in rows:
                zb[r // 2] |= (zz[r] << (4 * (r % 2))).astype(np.uint8)
            out[base + SB_NIB + SB_SCALE:base + SB_BYTES] = zb
    return out


def unrepack(buf, N, K, group=GROUP):
    """Inverse of repack(): interleaved bytes -> canonical (Q, S, Z).
    group 256: the scale and zero point of each group are read from its
    first super-block."""
    _check_layout(K, group)
    if group == 64:
        return _unrepack_g64(buf, N, K)
    if group != GROUP:
        Q, S, Z = unrepack(buf, N, K, GROUP)
        r = group // GROUP
        return Q, S[:, ::r].copy(), pack_zeros(unpack_zeros(Z, K // GROUP)[:, ::r])
    G = K // group
    Np = -(-N // ROW_TILE) * ROW_TILE
    buf = np.asarray(buf, np.uint8)
    q = np.zeros((Np, K), np.uint8)
    s = np.zeros((Np, G), np.uint16)
    z = np.zeros((Np, G), np.uint8)
    rows = np.arange(ROW_TILE)
    boff, half = _nibble_address(np.arange(GROUP)[None, :], rows[:, None])
    for T in range(Np // ROW_TILE):
        for g in range(G):
            base = (T * G + g) * SB_BYTES
            nib = buf[base:base + SB_NIB].reshape(ROW_TILE, 64)
            for kk in range(GROUP):
                q[T * ROW_TILE:(T + 1) * ROW_TILE, g * group + kk] = (nib[rows, boff[:, kk]] >> (4 * half[:, kk])) & 0xF
            s[T * ROW_TILE:(T + 1) * ROW_TILE, g] = buf[base + SB_NIB:base + SB_NIB + SB_SCALE].view('<u2')
            zb = buf[base + SB_NIB + SB_SCALE:base + SB_BYTES]
            z[T * ROW_TILE:(T + 1) * ROW_TILE, g] = (zb[rows // 2] >> (4 * (rows % 2))) & 0xF
    return pack_codes(q[:N]), s[:N].copy(), pack_zeros(z[:N])


def _repack_g64(Q, S, Z, N, K):
    """Groups of 64: the super-blocks of the 128-column layout carry the
    scale and zero point of the even group (columns 0..63 of the 128); the
    side array that follows them, one 320-byte entry per super-block in the
    same order, carries those of the odd group (columns 64..127): 128 fp16
    scales (row r at 2r, little endian), then 128 zero points (row r in byte
    256 + r//2, low nibble = even r)."""
    G64 = K // 64
    z = unpack_zeros(Z, G64)
    main = repack(Q, S[:, 0::2].copy(), pack_zeros(z[:, 0::2]), N, K, GROUP)
    Np = -(-N // ROW_TILE) * ROW_TILE
    nsb = (Np // ROW_TILE) * (K // GROUP)
    side = np.zeros(nsb * SB_SIDE, np.uint8)
    s_odd = np.zeros((Np, K // GROUP), np.uint16)
    s_odd[:N] = S[:, 1::2]
    z_odd = np.zeros((Np, K // GROUP), np.uint8)
    z_odd[:N] = z[:, 1::2]
    rows = np.arange(ROW_TILE)
    for u in range(nsb):
        T, g = divmod(u, K // GROUP)
        e = side[u * SB_SIDE:(u + 1) * SB_SIDE]
        e[:256] = s_odd[T * ROW_TILE:(T + 1) * ROW_TILE, g].astype('<u2').view(np.uint8)
        zz = z_odd[T * ROW_TILE:(T + 1) * ROW_TILE, g]
        for r in rows:
            e[256 + r // 2] |= (zz[r] << (4 * (r % 2))).astype(np.uint8)
    return np.concatenate([main, side])


def _unrepack_g64(buf, N, K):
    """Inverse of _repack_g64."""
    Np = -(-N // ROW_TILE) * ROW_TILE
    nsb = (Np // ROW_TILE) * (K // GROUP)
    buf = np.asarray(buf, np.uint8)
    Q, S_even, Z_even = unrepack(buf[:nsb * SB_BYTES], N, K, GROUP)
    S = np.zeros((N, K // 64), np.uint16)
    z = np.zeros((N, K // 64), np.uint8)
    S[:, 0::2] = S_even
    z[:, 0::2] = unpack_zeros(Z_even, K // GROUP)
    side = buf[nsb * SB_BYTES:]
    rows = np.arange(ROW_TILE)
    s_odd = np.zeros((Np, K // GROUP), np.uint16)
    z_odd = np.zeros((Np, K // GROUP), np.uint8)
    for u in range(nsb):
        T, g = divmod(u, K // GROUP)
        e = side[u * SB_SIDE:(u + 1) * SB_SIDE]
        s_odd[T * ROW_TILE:(T + 1) * ROW_TILE, g] = e[:256].view('<u2')
        z_odd[T * ROW_TILE:(T + 1) * ROW_TILE, g] = (e[256 + rows // 2] >> (4 * (rows % 2))) & 0xF
    S[:, 1::2] = s_odd[:N]
    z[:, 1::2] = z_odd[:N]
    return Q, S, pack_zeros(z)


# --------------------------------------------------------------------------
# f2: router projection
# --------------------------------------------------------------------------

def router_logits(x, w_router):
    """Router logits of the routed MoE layer, logits[m, e] = sum_h x[m, h] *
    Wr[e, h], in double (x float64 [M, H], Wr float64 [E, H]).  The pages
    give no detail of the router (the fastllm README only sets top-k, section
    "5. 其它参数"); the plain dense projection is the reading taken.  Returns
    (logits, tol) with the linear bound tol = 2e-3 * sum_h |x||Wr| + 1e-5 of
    an fp32-accumulated result."""
    x = np.asarray(x, np.float64)
    w = np.asarray(w_router, np.float64)
    return x @ w.T, 2e-3 * (np.abs(x) @ np.abs(w).T) + 1e-5


# --------------------------------------------------------------------------
# a5: routing and permutation
# --------------------------------------------------------------------------

SOFTMAX = 0
SIGMOID = 1


def route(logits, k, scoring=SOFTMAX, renorm=True, bias=None, n_group=1, topk_group=1, scale=1.0):
    """Top-k routing of fp32 router logits [M, E].

    bias / n_group > 1 (sigmoid scoring only) select the DeepSeek-V3 way,
    see route_keyed(); scale multiplies the final weights in every mode.

    Selection uses the raw fp32 logits: the k largest; equal logits go to
    the lower expert index; slots are ordered by descending logit, then
    ascending index.  Weights, in double:
      softmax: w_j = exp(l_j - l_max) / sum_sel exp(l - l_max) when renorm,
               else divided by the sum over all E (plain softmax);
      sigmoid: w_j = sigma(l_j) / sum_sel sigma(l) when renorm, else sigma(l_j).
    Returns ids int32 [M, k], weights float64 [M, k].
    """
    logits = np.asarray(logits, np.float32)
    M, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    if np.isnan(logits).any():
        raise ValueError("NaN router logit")
    ids = np.zeros((M, k), np.int32)
    wts = np.zeros((M, k), np.float64)
    for t in range(M):
        l = logits[t].astype(np.float64)
        order = sorted(range(E), key=lambda e: (-l[e], e))
        sel = np.array(order[:k])
        ids[t] = sel
        if scoring == SOFTMAX:
            lmax = l[sel[0]]
            ex = np.exp(l[sel] - lmax)
            den = ex.sum() if renorm else np.exp(l - lmax).sum()
            wts[t] = ex / den
        elif scoring == SIGMOID:
            sg = 1.0 / (1.0 + np.exp(-l[sel]))
            wts[t] = sg / sg.sum() if renorm else sg
        else:
            raise ValueError("unknown scoring")
    if bias is not None or n_group > 1:
        if scoring != SIGMOID:
            raise ValueError("the score bias and group-limited routing take sigmoid scoring")
        ids, wts = route_keyed(logits, k, renorm, bias, n_group, topk_group)
    return ids, wts * float(scale)


def route_keyed(logits, k, renorm=True, bias=None, n_group=1, topk_group=1):
    """DeepSeek-V3 style selection (sigmoid affinities, auxiliary-loss-free
    bias, group-limited experts), in double; not on the FastLLM pages, whose
    MoE options only fix top-k and the shared expert.

      s_e   = sigma(l_e)                         affinity (l: the fp32 logit)
      key_e = s_e + b_e                          b: fp32 bias, used for the choice only
      groups: n_group runs of E/n_group consecutive experts; a group's score is
              the sum of its two largest keys (its one key if it has one);
              the topk_group best groups are kept (ties: lower group index)
      experts: the k largest keys among the kept groups' experts (ties: lower
              index), slots ordered by descending key, then index
      w_j   = s_{e_j} / sum_sel s (renorm) or s_{e_j}: the bias is not in the weights
    """
    logits = np.asarray(logits, np.float32)
    M, E = logits.shape
    if n_group < 1 or E % n_group or not (1 <= topk_group <= n_group):
        raise ValueError("need E % n_group == 0 and 1 <= topk_group <= n_group")
    gsz = E // n_group
    if not (1 <= k <= topk_group * gsz):
        raise ValueError("need 1 <= k <= topk_group * E / n_group")
    b = np.zeros(E) if bias is None else np.asarray(bias, np.float32).astype(np.float64)
    ids = np.zeros((M, k), np.int32)
    wts = np.zeros((M, k), np.float64)
    for t in range(M):
        s = 1.0 / (1.0 + np.exp(-logits[t].astype(np.float64)))
        key = s + b
        gscore = []
        for g in range(n_group):
            kg = sorted(key[g * gsz:(g + 1) * gsz], reverse=True)
            gscore.append(sum(kg[:2]))
        kept = sorted(range(n_group), key=lambda g: (-gscore[g], g))[:topk_group]
        eligible = [e for e in range(E) if e // gsz in kept]
        sel = sorted(eligible, key=lambda e: (-key[e], e))[:k]
        ids[t] = sel
        sg = s[sel]
        wts[t] = sg / sg.sum() if renorm else sg
    return ids, wts


def permute(ids, E):
    """Stable counting sort of the flattened assignments t*k + j by expert.

    Returns (expert_offsets int32 [E+1] -- exclusive scan of per-expert
    counts, perm int32 [M*k] -- perm[pos] = t*k + j, experts ascending and,
    within an expert, flattened index ascending).
    """
    flat = np.asarray(ids, np.int64).reshape(-1)
    counts = np.array([(flat == e).sum() for e in range(E)], np.int64)
    offsets = np.zeros(E + 1, np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.zeros(flat.size, np.int64)
    fill = offsets[:-1].copy()
    for i in range(flat.size):          # visiting i in order keeps it stable
        e = flat[i]
        perm[fill[e]] = i
        fill[e] += 1
    return offsets.astype(np.int32), perm.astype(np.int32)


# --------------------------------------------------------------------------
# a6/a7: expert FFN, combine, error bound
# --------------------------------------------------------------------------

def silu(a):
    with np.errstate(over='ignore'):
        return a / (1.0 + np.exp(-a))


def silu_grad(a):
    with np.errstate(over='ignore'):
        sg = 1.0 / (1.0 + np.exp(-a))
    return sg * (1.0 + a * (1.0 - sg))


def expert_ffn(x, w13, w2, group=GROUP):
    """One expert on tokens x float64 [T, H].

    w13 = (Q, S, Z) of [2I, H]: rows 0..I-1 gate, rows I..2I-1 up.
    w2  = (Q, S, Z) of [H, I].
    h = silu(G x) * (U x);  out = W2 h.
    Returns (out [T, H], tol_out [T, H]) where tol_out bounds, to first
    order, the error of a path that computes both projections to the linear
    bound (2e-3 relative to sum |a||w'|, fp32 accumulation) and stores h in
    bf16 (the worst case of that error model reaches it up to second-order
    terms: products of two moves and the curvature of silu):
      tol_h = 2e-3 (|silu'(g)| A_g |u| + |silu(g)| A_u) + 2^-8 |h|
      tol_out = 2e-3 |h| |W2'|^T + tol_h |W2'|^T
    """
    W13 = dequantize(*w13, group=group)
    W2 = dequantize(*w2, group=group)
    I = W13.shape[0] // 2
    x = np.asarray(x, np.float64)
    gu = x @ W13.T
    A = np.abs(x) @ np.abs(W13).T
    g, u = gu[:, :I], gu[:, I:]
    Ag, Au = A[:, :I], A[:, I:]
    h = silu(g) * u
    tol_h = 2e-3 * (np.abs(silu_grad(g)) * Ag * np.abs(u) + np.abs(silu(g)) * Au) + BF16_U * np.abs(h)
    out = h @ W2.T
    tol = 2e-3 * (np.abs(h) @ np.abs(W2).T) + tol_h @ np.abs(W2).T
    return out, tol


def moe(x, logits, k, w13, w2, scoring=SOFTMAX, renorm=True,
        shared_w13=None, shared_w2=None, group=GROUP, routing=None):
    """Routed MoE layer with int4g experts, in double.

    x float64 [M, H]; logits fp32 [M, E]; w13[e], w2[e] canonical triples
    (any indexable, fetched only for experts that receive tokens).
    y[t] = sum_j w_{t,j} * expert_{ids[t,j]}(x[t])  (+ shared(x[t]) * 1).
    Returns (y, tol, ids, weights) with tol the propagated elementwise bound
    (the per-expert bound above, weighted by the gate weights, + 1e-5),
    widened by the final bf16 store of y.
    """
    x = np.asarray(x, np.float64)
    M, H = x.shape
    ids, wts = route(logits, k, scoring, renorm, **(routing or {}))
    y = np.zeros((M, H))
    tol = np.zeros((M, H))
    for e in np.unique(ids):
        tok, slot = np.nonzero(ids == e)
        out, t_out = expert_ffn(x[tok], w13[e], w2[e], group)
        wv = wts[tok, slot][:, None]
        for i in range(tok.size):      # a token meets an expert at most once
            y[tok[i]] += wv[i] * out[i]
            tol[tok[i]] += wv[i] * t_out[i]
    if shared_w13 is not None:
        out, t_out = expert_ffn(x, shared_w13, shared_w2, group)
        y += out
        tol += t_out
    return y, _with_output_rounding(tol + 1e-5, y), ids, wts
