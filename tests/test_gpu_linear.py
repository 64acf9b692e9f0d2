"""GPU parity: quantizer, repack and int4g linear through the C ABI against
the CPU oracle on the same seeded inputs.

Bar: codes, scales, zeros and the interleaved bytes bit-exact; y within
|y - y_ref| <= 2e-3 * sum_k |x||w'| + 1e-5 elementwise (fp32 accumulation,
bf16 output)."""
import numpy as np
import pytest
import torch

import int4_group_quantized_int4g_gb300 as fl
from int4_group_quantized_int4g_gb300 import inputs
from oracle import int4g_oracle as O

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from int4_group_quantized_int4g_gb300 import _build
    _build.build()
    fl.lib()


def to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bf16_dev(bits):
    return to_dev(bits.view(np.int16)).view(torch.bfloat16)


def quantize_dev(W):
    q, s, z = fl.fl_int4g_quantize(to_dev(W))
    return q, s, z


def canon_host(q, s, z):
    return q.cpu().numpy(), s.cpu().numpy().view(np.uint16), z.cpu().numpy()


# ------------------------------------------------------------ a1 quantizer

def _edge_weights():
    rng = np.random.default_rng([0, 40])
    W = (rng.standard_normal((7, 1024)) * 0.02).astype(np.float32)
    W[0, 0:128] = 0.0                          # zero group
    W[0, 128:256] = 0.37                       # constant positive
    W[0, 256:384] = -1.25                      # constant negative
    W[1, 0:128] = np.float32(1e-9) * rng.standard_normal(128).astype(np.float32)   # s16 -> 0
    W[1, 128:256] = np.float32(3e-6) * rng.standard_normal(128).astype(np.float32)  # fp16 subnormal scale
    W[2, 0:128] = np.abs(W[2, 0:128]) + 0.5    # all positive: clamped zero point
    W[2, 128:256] = -np.abs(W[2, 128:256]) - 0.5
    # exact rounding ties: on a grid with step 0.25 plus half steps
    W[3, 0:128] = (np.arange(128) % 16 - 7.5).astype(np.float32) * np.float32(0.25)
    W[4, :] *= 50                              # large values
    return W


@pytest.mark.parametrize("shape", [(200, 384), (3, 1024), (129, 1152)])
def test_quantizer_bit_exact(shape):
    N, K = shape
    W = inputs.dense_weight(N, K, layer=40 + N)
    Q, S, Z = O.quantize(W)
    got = canon_host(*quantize_dev(W))
    assert np.array_equal(got[0], Q)
    assert np.array_equal(got[1], S)
    assert np.array_equal(got[2], Z)


def test_quantizer_edge_groups_bit_exact():
    W = _edge_weights()
    Q, S, Z = O.quantize(W)
    got = canon_host(*quantize_dev(W))
    assert np.array_equal(got[0], Q) and np.array_equal(got[1], S) and np.array_equal(got[2], Z)


def test_quantizer_reports_fp16_overflow():
    W = np.zeros((2, 256), np.float32)
    W[1, 130] = 4e6
    W[1, 131] = -4e6
    with pytest.raises(fl.Int4gError) as e:
        quantize_dev(W)
    assert e.value.code == 7


# ------------------------------------------------------------ a2 repack

@pytest.mark.parametrize("shape", [(200, 384), (128, 128), (300, 1280)])
def test_repack_bit_exact_and_invertible(shape):
    N, K = shape
    W = inputs.dense_weight(N, K, layer=50 + N)
    Q, S, Z = O.quantize(W)
    w = fl.fl_int4g_repack(to_dev(Q), to_dev(S.view(np.int16)), to_dev(Z), N, K)
    assert np.array_equal(w.cpu().numpy(), O.repack(Q, S, Z, N, K))
    back = canon_host(*fl.fl_int4g_unrepack(w, N, K))
    assert np.array_equal(back[0], Q) and np.array_equal(back[1], S) and np.array_equal(back[2], Z)


# ------------------------------------------------- groups of 256 (a1, a2, a3)
# FastLLM page, section 4.2: --group-size 128 by default, 256 allowed.  The
# interleaved layout keeps 128-column super-blocks; both super-blocks of a
# group carry its scale and zero point, so the matmul kernels are unchanged.

@pytest.mark.parametrize("shape", [(200, 512), (3, 1024), (129, 1280)])
def test_quantizer_group256_bit_exact(shape):
    N, K = shape
    W = inputs.dense_weight(N, K, layer=80 + N)
    W[0, :256] = 0.0             # zero group
    W[1 % N, 256:512] = -0.75    # constant negative group
    Q, S, Z = O.quantize(W, 256)
    got = canon_host(*fl.fl_int4g_quantize(to_dev(W), group=256))
    assert np.array_equal(got[0], Q)
    assert np.array_equal(got[1], S)
    assert np.array_equal(got[2], Z)


@pytest.mark.parametrize("shape", [(200, 512), (128, 256), (300, 1280)])
def test_repack_group256_bit_exact_and_invertible(shape):
    N, K = shape
    W = inputs.dense_weight(N, K, layer=90 + N)
    Q, S, Z = O.quantize(W, 256)
    w = fl.fl_int4g_repack(to_dev(Q), to_dev(S.view(np.int16)), to_dev(Z), N, K, group=256)
    assert np.array_equal(w.cpu().numpy(), O.repack(Q, S, Z, N, K, 256))
    back = canon_host(*fl.fl_int4g_unrepack(w, N, K, group=256))
    assert np.array_equal(back[0], Q) and np.array_equal(back[1], S) and np.array_equal(back[2], Z)


# Groups of 64 (FastLLM page, section 5.4): the super-blocks carry the even
# group's scale and zero point, a side array after them the odd group's.

@pytest.mark.parametrize("shape", [(200, 384), (3, 1024), (129, 1280)])
def test_quantizer_group64_bit_exact(shape):
    N, K = shape
    W = inputs.dense_weight(N, K, layer=70 + N)
    W[0, :64] = 0.0              # zero group
    W[1 % N, 64:128] = 0.5       # constant positive group
    W[2 % N, 128:192] = np.abs(W[2 % N, 128:192]) + 0.25   # all positive: clamped zero point
    Q, S, Z = O.quantize(W, 64)
    got = canon_host(*fl.fl_int4g_quantize(to_dev(W), group=64))
    assert np.array_equal(got[0], Q)
    assert np.array_equal(got[1], S)
    assert np.array_equal(got[2], Z)


@pytest.mark.parametrize("shape", [(200, 384), (128, 128), (300, 1280)])
def test_repack_group64_bit_exact_and_invertible(shape):
    N, K = shape
    W = inputs.dense_weight(N, K, layer=60 + N)
    Q, S, Z = O.quantize(W, 64)
    w = fl.fl_int4g_repack(to_dev(Q), to_dev(S.view(np.int16)), to_dev(Z), N, K, group=64)
    assert np.array_equal(w.cpu().numpy(), O.repack(Q, S, Z, N, K, 64))
    back = canon_host(*fl.fl_int4g_unrepack(w, N, K, group=64))
    assert np.array_equal(back[0], Q) and np.array_equal(back[1], S) and np.array_equal(back[2], Z)


@pytest.mark.parametrize("M", [1, 5, 8, 9, 16, 32, 33, 64, 300])
@pytest.mark.parametrize("NK", [(384, 1280), (200, 256)])
def test_linear_group64_parity(M, NK):
    """Decode (the mma.sync kernel, one accumulator per 64-column group) and
    prefill (the tcgen05 GEMM, each K half dequantized with its own group's
    scale) on group-64 weights quantized and repacked on the GPU, against
    the oracle's group-64 linear, every output."""
    N, K = NK
    W = inputs.dense_weight(N, K, layer=40 + M + N)
    Q, S, Z = O.quantize(W, 64)
    q, s_, z = fl.fl_int4g_quantize(to_dev(W), group=64)
    w = fl.fl_int4g_repack(q, s_, z, N, K, group=64)
    xb = inputs.activations(M, K, stream=40 + M)
    y = fl.fl_int4g_linear(bf16_dev(xb), w, N, group=64)
    xf = O.bf16_value(xb)
    ref, tol = O.linear(xf, Q, S, Z, 64), O.linear_tolerance(xf, Q, S, Z, 64)
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= tol), f"worst err/tol {np.max(np.abs(got - ref) / tol):.3f}"
    # the groups of 64 matter: the same codes read as groups of 128 (the even
    # groups' scales only) give a different result
    y128 = fl.fl_int4g_linear(bf16_dev(xb), w, N)
    assert not torch.equal(y.view(torch.int16), y128.view(torch.int16))


def test_linear_group64_llama_sampled():
    """K=4096, N=11008 at M in {1, 8, 32, 512}: 64 sampled columns."""
    K, N = 4096, 11008
    W = inputs.dense_weight(N, K, layer=64064)
    q, s_, z = fl.fl_int4g_quantize(to_dev(W), group=64)
    w = fl.fl_int4g_repack(q, s_, z, N, K, group=64)
    cols = np.unique(np.concatenate([np.sort(inputs.rng(9, K, N).choice(N, 64, replace=False)), [0, N - 1]]))
    Qc, Sc, Zc = O.quantize(W[cols], 64)
    for M in (1, 8, 32, 512):
        xb = inputs.activations(M, K, stream=M + 64)
        y = fl.fl_int4g_linear(bf16_dev(xb), w, N, group=64)
        xf = O.bf16_value(xb)
        ref, tol = O.linear(xf, Qc, Sc, Zc, 64), O.linear_tolerance(xf, Qc, Sc, Zc, 64)
        got = y.float().cpu().numpy().astype(np.float64)[:, cols]
        assert np.all(np.abs(got - ref) <= tol), (M, np.max(np.abs(got - ref) / tol))


def test_linear_group64_long_k_many_tokens():
    """Groups of 64 at M=32 with K=28672 (N=7168): the decode kernel's plan
    would take ten 19 KB stages and overflow the 227 KB shared-memory limit;
    it runs with nine.  64 sampled columns, the first and the last among
    them, against the oracle's group-64 linear."""
    M, K, N = 32, 28672, 7168
    W = inputs.dense_weight(N, K, layer=64065)
    q, s_, z = fl.fl_int4g_quantize(to_dev(W), group=64)
    w = fl.fl_int4g_repack(q, s_, z, N, K, group=64)
    cols = np.unique(np.concatenate([np.sort(inputs.rng(10, K, N).choice(N, 64, replace=False)), [0, N - 1]]))
    Qc, Sc, Zc = O.quantize(W[cols], 64)
    del W
    xb = inputs.activations(M, K, stream=M + 65)
    y = fl.fl_int4g_linear(bf16_dev(xb), w, N, group=64)
    xf = O.bf16_value(xb)
    ref, tol = O.linear(xf, Qc, Sc, Zc, 64), O.linear_tolerance(xf, Qc, Sc, Zc, 64)
    got = y.float().cpu().numpy().astype(np.float64)[:, cols]
    assert np.all(np.abs(got - ref) <= tol), np.max(np.abs(got - ref) / tol)


@pytest.mark.parametrize("M", [1, 8, 9, 32, 64, 300])
def test_linear_group256_parity(M):
    """Decode (rows and tcgen05 kernels) and prefill on group-256 weights,
    quantized and repacked on the GPU, against the oracle's group-256 linear."""
    N, K = 384, 1280
    W = inputs.dense_weight(N, K, layer=95)
    xb = inputs.activations(M, K, stream=95)
    Q, S, Z = O.quantize(W, 256)
    q, s, z = fl.fl_int4g_quantize(to_dev(W), group=256)
    w = fl.fl_int4g_repack(q, s, z, N, K, group=256)
    y = fl.fl_int4g_linear(bf16_dev(xb), w, N)
    xf = O.bf16_value(xb)
    ref, tol = O.linear(xf, Q, S, Z, 256), O.linear_tolerance(xf, Q, S, Z, 256)
    got = y.float().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= tol), f"worst err/tol {np.max(np.abs(got - ref) / tol):.3f}"


# ------------------------------------------------------------ a3 linear

def _linear_case(M, N, K, layer):
    W = inputs.dense_weight(N, K, layer=layer)
    xb = inputs.activations(M, K, stream=layer)
    Q, S, Z = O.quantize(W)
    w = fl.fl_int4g_repack(to_dev(Q), to_dev(S.view(np.int16)), to_dev(Z), N, K)
    return W, xb, Q, S, Z, w


def _check(y, xb, Q, S, Z):
    xf = O.bf16_value(xb)
    ref, tol = O.linear(xf, Q, S, Z), O.linear_tolerance(xf, Q, S, Z)
    got = y.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    bad = err > tol
    assert not bad.any(), f"{bad.sum()} elements out of bound; worst err/tol {np.max(err / tol):.3f} at {np.unravel_index(np.argmax(err / tol), err.shape)}"
    # aggregate sanity check beside the elementwise bound: relative RMS error
    # near the bf16 rounding floor of the output
    rel = np.sqrt(np.mean(err ** 2) / np.mean(ref ** 2))
    assert rel <= 1e-2, f"relative RMS error {rel:.3e}"
    return float(np.max(err / tol))


@pytest.mark.parametrize("M", [1, 2, 7, 8, 9, 16, 17, 31, 32, 33, 40])
@pytest.mark.parametrize("NK", [(200, 384), (512, 1280), (136, 128)])
def test_linear_parity_small(M, NK):
    N, K = NK
    _, xb, Q, S, Z, w = _linear_case(M, N, K, layer=60 + K)
    y = fl.fl_int4g_linear(bf16_dev(xb), w, N)
    _check(y, xb, Q, S, Z)


def test_linear_config1_full():
    """M=1, K=1024, N=3072 (Qwen3-0.6B up_proj shape), every output checked."""
    M, N, K = 1, 3072, 1024
    W = inputs.dense_weight(N, K, layer=0, outliers=False)
    xb = inputs.activations(M, K, stream=0)
    Q, S, Z = O.quantize(W)
    q, s, z = quantize_dev(W)
    assert np.array_equal(canon_host(q, s, z)[0], Q)
    w = fl.fl_int4g_repack(q, s, z, N, K)
    y = fl.fl_int4g_linear(bf16_dev(xb), w, N)
    _check(y, xb, Q, S, Z)


def test_linear_deterministic_and_workspace_reuse():
    M, N, K = 8, 1024, 4096
    _, xb, Q, S, Z, w = _linear_case(M, N, K, layer=70)
    x = bf16_dev(xb)
    y1 = fl.fl_int4g_linear(x, w, N).clone()
    y2 = fl.fl_int4g_linear(x, w, N).clone()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    _check(y1, xb, Q, S, Z)


def test_linear_workspace_too_small():
    M, N, K = 1, 256, 256
    _, xb, Q, S, Z, w = _linear_case(M, N, K, layer=71)
    ws = torch.zeros(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(fl.Int4gError) as e:
        fl.fl_int4g_linear(bf16_dev(xb), w, N, ws=ws)
    assert e.value.code == 2


LLAMA = [(4096, 12288), (4096, 11008), (11008, 4096)]


@pytest.mark.parametrize("KN", LLAMA)
def test_linear_llama_decode_sampled(KN):
    """Llama-7B-shaped decode linears at full size, M in {1, 8, 32}, on 96
    sampled output columns (the oracle dequantizes just those rows)."""
    K, N = KN
    W = inputs.dense_weight(N, K, layer=K + N)
    q, s, z = quantize_dev(W)
    w = fl.fl_int4g_repack(q, s, z, N, K)
    cols = np.sort(inputs.rng(6, K, N).choice(N, 96, replace=False))
    cols = np.unique(np.concatenate([cols, [0, N - 1]]))
    Qc, Sc, Zc = O.quantize(W[cols])
    qh, sh, zh = canon_host(q, s, z)
    assert np.array_equal(qh[cols], Qc) and np.array_equal(sh[cols], Sc) and np.array_equal(zh[cols], Zc)
    for M in (1, 8, 32):
        xb = inputs.activations(M, K, stream=M)
        y = fl.fl_int4g_linear(bf16_dev(xb), w, N)
        xf = O.bf16_value(xb)
        ref, tol = O.linear(xf, Qc, Sc, Zc), O.linear_tolerance(xf, Qc, Sc, Zc)
        got = y.float().cpu().numpy().astype(np.float64)[:, cols]
        assert np.all(np.abs(got - ref) <= tol), (M, np.max(np.abs(got - ref) / tol))
        assert np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2)) <= 1e-2


@pytest.mark.parametrize("M", [1, 8])
def test_linear_stream_k_many_row_tiles(M):
    """A vocabulary-sized decode linear (K=4096, N=32000: 250 row tiles, more
    than half the CTA slots) takes the stream-K split with the ticket
    hand-off instead of cluster reductions; 96 sampled columns, the first
    and the last, against the oracle."""
    K, N = 4096, 32000
    W = inputs.dense_weight(N, K, layer=N + M)
    q, s, z = quantize_dev(W)
    w = fl.fl_int4g_repack(q, s, z, N, K)
    cols = np.unique(np.concatenate([np.sort(inputs.rng(8, K, N).choice(N, 96, replace=False)), [0, N - 1]]))
    Qc, Sc, Zc = O.quantize(W[cols])
    xb = inputs.activations(M, K, stream=N + M)
    ws = torch.zeros(fl.fl_int4g_linear_workspace(M, N, K), dtype=torch.uint8, device=DEV)
    for _ in range(2):   # the tickets are left zero for the next call
        y = fl.fl_int4g_linear(bf16_dev(xb), w, N, ws=ws)
        xf = O.bf16_value(xb)
        ref, tol = O.linear_columns(xf, Qc, Sc, Zc, np.arange(len(cols)))
        got = y.float().cpu().numpy().astype(np.float64)[:, cols]
        assert np.all(np.abs(got - ref) <= tol), (M, np.max(np.abs(got - ref) / tol))
    assert fl.fl_int4g_status(ws) == 0


@pytest.mark.parametrize("M", [1, 8])
def test_linear_cluster_long_k(M):
    """A long-K decode linear (K=32768, N=1024: 8 row tiles, each split over
    a cluster of 8 ranks of 32 groups).  At M=1 each rank keeps the x rows of
    its K slice in an x region of shared memory; at M=8 that region (8 x 8 KB)
    would leave fewer than three weight stages, so x travels in the stages.
    66 sampled columns, the first and the last among them, against the
    oracle."""
    K, N = 32768, 1024
    W = inputs.dense_weight(N, K, layer=K + M)
    q, s, z = quantize_dev(W)
    w = fl.fl_int4g_repack(q, s, z, N, K)
    cols = np.unique(np.concatenate([np.sort(inputs.rng(9, K, N).choice(N, 64, replace=False)), [0, N - 1]]))
    Qc, Sc, Zc = O.quantize(W[cols])
    xb = inputs.activations(M, K, stream=K + M)
    y = fl.fl_int4g_linear(bf16_dev(xb), w, N)
    xf = O.bf16_value(xb)
    ref, tol = O.linear_columns(xf, Qc, Sc, Zc, np.arange(len(cols)))
    got = y.float().cpu().numpy().astype(np.float64)[:, cols]
    assert np.all(np.abs(got - ref) <= tol), (M, np.max(np.abs(got - ref) / tol))


def test_cluster_reduction_timeout_is_reported():
    """The failure path of the decode kernel's bounded inter-CTA wait, made
    to run out by the test hook (a barrier arrival nobody makes, 1 ms
    bound): the status block reports FL_ERR_TIMEOUT, the kernel returns (no
    hang, no fault), and the same workspace then serves a normal call."""
    M, N, K = 1, 200, 1024   # 2 row tiles: each split over K by a cluster of 8 CTAs
    _, xb, Q, S, Z, w = _linear_case(M, N, K, layer=72)
    x = bf16_dev(xb)
    ws = torch.zeros(fl.fl_int4g_linear_workspace(M, N, K), dtype=torch.uint8, device=DEV)
    fl.fl_int4g_test_withhold_cluster_arrival(1_000_000)
    try:
        fl.fl_int4g_linear(x, w, N, ws=ws)
        torch.cuda.synchronize()
    finally:
        fl.fl_int4g_test_withhold_cluster_arrival(-1)
    assert fl.fl_int4g_status(ws) == 5
    y = fl.fl_int4g_linear(x, w, N, ws=ws)
    _check(y, xb, Q, S, Z)
    assert fl.fl_int4g_status(ws) == 0


def test_linear_one_workspace_across_shapes():
    """One workspace serves shapes with different tile counts in turn: a call
    must not find the previous shape's scratch where its counters are."""
    shapes = [(32, 512, 1280), (1, 3072, 1024), (8, 200, 384), (32, 1024, 2048), (1, 3072, 1024)]
    nb = max(fl.fl_int4g_linear_workspace(M, N, K) for (M, N, K) in shapes)
    ws = torch.zeros(nb, dtype=torch.uint8, device=DEV)
    for i, (M, N, K) in enumerate(shapes):
        _, xb, Q, S, Z, w = _linear_case(M, N, K, layer=80 + i)
        y = fl.fl_int4g_linear(bf16_dev(xb), w, N, ws=ws)
        _check(y, xb, Q, S, Z)
    assert fl.fl_int4g_status(ws) == 0


# ------------------------------------------------------------ a4 prefill (tcgen05)

@pytest.mark.parametrize("M", [33, 64, 127, 128, 129, 300, 1000, 1100])
@pytest.mark.parametrize("NK", [(200, 384), (384, 1280)])
def test_prefill_parity_small(M, NK):
    N, K = NK
    _, xb, Q, S, Z, w = _linear_case(M, N, K, layer=90 + K)
    y = fl.fl_int4g_linear(bf16_dev(xb), w, N)
    _check(y, xb, Q, S, Z)


@pytest.mark.parametrize("KN", [(4096, 11008), (11008, 4096)])
def test_prefill_full_size_sampled(KN):
    """Prefill shapes M in {512, 2048} at full size, 64 sampled output columns
    (all tokens) against the oracle."""
    K, N = KN
    W = inputs.dense_weight(N, K, layer=K + N + 1)
    q, s, z = quantize_dev(W)
    w = fl.fl_int4g_repack(q, s, z, N, K)
    cols = np.unique(np.concatenate([np.sort(inputs.rng(7, K, N).choice(N, 64, replace=False)), [0, N - 1]]))
    Qc, Sc, Zc = O.quantize(W[cols])
    for M in (512, 2048):
        xb = inputs.activations(M, K, stream=M + 1)
        y = fl.fl_int4g_linear(bf16_dev(xb), w, N)
        xf = O.bf16_value(xb)
        ref, tol = O.linear_columns(xf, Qc, Sc, Zc, np.arange(len(cols)))
        got = y.float().cpu().numpy().astype(np.float64)[:, cols]
        assert np.all(np.abs(got - ref) <= tol), (M, np.max(np.abs(got - ref) / tol))
        assert np.sqrt(np.mean((got - ref) ** 2) / np.mean(ref ** 2)) <= 1e-2


def test_one_workspace_across_entry_points():
    """One workspace serves the linear, the MoE layer, the router projection
    and the MLP block in turn: every entry point keeps its scratch out of the
    counter region that the others need zero."""
    M, N, K = 12, 512, 1280
    _, xb, Q, S, Z, w = _linear_case(M, N, K, layer=85)
    E, H, I = 8, 256, 128
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device=DEV)
    x = bf16_dev(xb)
    y0 = fl.fl_int4g_linear(x, w, N, ws=ws).clone()
    w13 = torch.cat([fl.fl_int4g_repack(*quantize_dev(inputs.expert_weight(2 * I, H, 86, e, 0)), 2 * I, H)
                     for e in range(E)])
    w2 = torch.cat([fl.fl_int4g_repack(*quantize_dev(inputs.expert_weight(H, I, 86, e, 1)), H, I) for e in range(E)])
    xm = bf16_dev(inputs.activations(40, H, stream=86))
    fl.fl_moe_int4g(xm, to_dev(inputs.router_logits(40, E, stream=86)), 2, I, w13, w2, ws=ws)
    wr = bf16_dev(inputs.to_bf16_bits(inputs.expert_weight(E, H, 87, 0, 0)))
    fl.fl_moe_router_logits(xm, wr, ws=ws)
    g, u, d = (fl.fl_int4g_repack(*quantize_dev(inputs.dense_weight(n, k, layer=88 + i)), n, k)
               for i, (n, k) in enumerate([(I, H), (I, H), (H, I)]))
    fl.fl_int4g_mlp(xm[:4].contiguous(), g, u, d, I, ws=ws)
    for _ in range(2):
        y = fl.fl_int4g_linear(x, w, N, ws=ws)
        assert torch.equal(y.view(torch.int16), y0.view(torch.int16))
    assert fl.fl_int4g_status(ws) == 0
    _check(y0, xb, Q, S, Z)
