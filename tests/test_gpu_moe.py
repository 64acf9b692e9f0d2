"""GPU parity of the routed MoE layer (route, permute, grouped gate/up +
SwiGLU, grouped down, weighted combine, shared expert) through the C ABI
against the CPU oracle on the same seeded inputs.

Bar: top-k ids, expert offsets and the permutation bit-exact; gate weights
within 1e-5 relative; y within the oracle's propagated elementwise bound."""
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


def repack_dev(Q, S, Z, N, K):
    return fl.fl_int4g_repack(to_dev(Q), to_dev(S.view(np.int16)), to_dev(Z), N, K)


def host_experts(E, H, I, layer):
    """Canonical triples (oracle quantizer) of E experts; numpy weights."""
    w13, w2 = [], []
    for e in range(E):
        w13.append(O.quantize(inputs.expert_weight(2 * I, H, layer, e, 0)))
        w2.append(O.quantize(inputs.expert_weight(H, I, layer, e, 1)))
    return w13, w2


def stack_dev(trips, N, K):
    return torch.cat([repack_dev(*t, N, K) for t in trips])


def run_moe(xb, logits, k, I, w13_d, w2_d, scoring, renorm, sw13=None, sw2=None):
    M, H = xb.shape
    E = logits.shape[1]
    ids = torch.empty((M, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((M, k), dtype=torch.float32, device=DEV)
    offs = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(M * k, dtype=torch.int32, device=DEV)
    ws = torch.zeros(fl.fl_moe_int4g_workspace(M, E, k, H, I, sw13 is not None), dtype=torch.uint8, device=DEV)
    y = fl.fl_moe_int4g(bf16_dev(xb), to_dev(logits), k, I, w13_d, w2_d, scoring=scoring, renorm=renorm,
                        shared_w13=sw13, shared_w2=sw2, topk_ids=ids, topk_w=wts, expert_offsets=offs, perm=perm,
                        ws=ws)
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 0
    return y, ids, wts, offs, perm


def check_y(y, ref, tol, rows=None):
    """The elementwise bound, plus an aggregate check: the propagated MoE bound
    is loose (first-order worst case), so the relative RMS error must also stay
    near the bf16 rounding floor of the output (~2.4e-3 observed)."""
    got = y.float().cpu().numpy().astype(np.float64)
    if rows is not None:
        got = got[rows]
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), f"worst err/tol {np.max(err / tol):.3f} at {np.unravel_index(np.argmax(err / tol), err.shape)}"
    rel = np.sqrt(np.mean(err ** 2) / np.mean(ref ** 2))
    assert rel <= 1e-2, f"relative RMS error {rel:.3e}"


def check_routing(logits, k, scoring, renorm, ids, wts, offs, perm):
    E = logits.shape[1]
    rid, rw = O.route(logits, k, scoring, renorm)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(wts.cpu().numpy(), rw, rtol=1e-5, atol=1e-7)
    roff, rperm = O.permute(rid, E)
    assert np.array_equal(offs.cpu().numpy(), roff)
    assert np.array_equal(perm.cpu().numpy(), rperm)


@pytest.fixture(scope="module")
def small():
    E, H, I = 8, 256, 256
    w13, w2 = host_experts(E, H, I, layer=500)
    sw13, sw2 = host_experts(1, H, I, layer=501)
    return dict(E=E, H=H, I=I, w13=w13, w2=w2, sw13=sw13[0], sw2=sw2[0],
                w13_d=stack_dev(w13, 2 * I, H), w2_d=stack_dev(w2, H, I),
                sw13_d=repack_dev(*sw13[0], 2 * I, H), sw2_d=repack_dev(*sw2[0], H, I))


@pytest.mark.parametrize("M", [1, 5, 8, 9, 37, 70])
@pytest.mark.parametrize("mode", ["softmax", "sigmoid_shared", "softmax_norenorm"])
def test_moe_small_parity(small, M, mode):
    E, H, I = small["E"], small["H"], small["I"]
    k = 3
    xb = inputs.activations(M, H, stream=600 + M)
    logits = inputs.router_logits(M, E, stream=600 + M)
    scoring = fl.FL_SIGMOID if mode.startswith("sigmoid") else fl.FL_SOFTMAX
    renorm = mode != "softmax_norenorm"
    shared = mode.endswith("shared")
    y, ids, wts, offs, perm = run_moe(xb, logits, k, I, small["w13_d"], small["w2_d"], scoring, renorm,
                                      small["sw13_d"] if shared else None, small["sw2_d"] if shared else None)
    check_routing(logits, k, scoring, renorm, ids, wts, offs, perm)
    ref, tol, _, _ = O.moe(O.bf16_value(xb), logits, k, small["w13"], small["w2"], scoring, renorm,
                           small["sw13"] if shared else None, small["sw2"] if shared else None)
    check_y(y, ref, tol)


def test_moe_routing_ties_and_all_experts(small):
    """Tied logits (quarter steps) and k = E: ids and permutation bit-exact."""
    E, H, I = small["E"], small["H"], small["I"]
    M = 33
    rng = np.random.default_rng([0, 610])
    logits = (np.round(rng.standard_normal((M, E)) * 2) / 4).astype(np.float32)
    xb = inputs.activations(M, H, stream=610)
    for k in (2, E):
        y, ids, wts, offs, perm = run_moe(xb, logits, k, I, small["w13_d"], small["w2_d"], fl.FL_SOFTMAX, True)
        check_routing(logits, k, fl.FL_SOFTMAX, True, ids, wts, offs, perm)
        ref, tol, _, _ = O.moe(O.bf16_value(xb), logits, k, small["w13"], small["w2"], O.SOFTMAX, True)
        check_y(y, ref, tol)


@pytest.mark.parametrize("M", [8, 9])
def test_moe_full_segments(small, M):
    """Every token routed to the same k experts: at M = 8 each of them holds
    one full segment of 8 positions, at M = 9 two segments (8 and 1)."""
    E, H, I = small["E"], small["H"], small["I"]
    k = 3
    row = inputs.router_logits(1, E, stream=630)
    logits = np.repeat(row, M, axis=0)
    xb = inputs.activations(M, H, stream=630 + M)
    y, ids, wts, offs, perm = run_moe(xb, logits, k, I, small["w13_d"], small["w2_d"], fl.FL_SIGMOID, True,
                                      small["sw13_d"], small["sw2_d"])
    check_routing(logits, k, fl.FL_SIGMOID, True, ids, wts, offs, perm)
    assert sorted(np.diff(offs.cpu().numpy()).tolist())[-k:] == [M] * k
    ref, tol, _, _ = O.moe(O.bf16_value(xb), logits, k, small["w13"], small["w2"], O.SIGMOID, True,
                           small["sw13"], small["sw2"])
    check_y(y, ref, tol)


@pytest.mark.parametrize("M", [12, 24])
def test_moe_segments_of_8_past_decode(M):
    """Up to 4 positions per expert on average, M > 8: segments of 8 built by
    the permute kernel (an expert with more than 8 positions spans two)."""
    E, H, I, k = 32, 256, 256, 4
    w13, w2 = host_experts(E, H, I, layer=640)
    sw13, sw2 = host_experts(1, H, I, layer=641)
    xb = inputs.activations(M, H, stream=640 + M)
    logits = inputs.router_logits(M, E, stream=640 + M)
    logits[:, 3] += 4.0   # one expert chosen by every token: M > 8 positions
    y, ids, wts, offs, perm = run_moe(xb, logits, k, I, stack_dev(w13, 2 * I, H), stack_dev(w2, H, I),
                                      fl.FL_SIGMOID, True, repack_dev(*sw13[0], 2 * I, H), repack_dev(*sw2[0], H, I))
    check_routing(logits, k, fl.FL_SIGMOID, True, ids, wts, offs, perm)
    assert np.diff(offs.cpu().numpy())[3] == M
    ref, tol, _, _ = O.moe(O.bf16_value(xb), logits, k, w13, w2, O.SIGMOID, True, sw13[0], sw2[0])
    check_y(y, ref, tol)


def test_moe_deterministic(small):
    M = 37
    xb = inputs.activations(M, small["H"], stream=620)
    logits = inputs.router_logits(M, small["E"], stream=620)
    a = run_moe(xb, logits, 3, small["I"], small["w13_d"], small["w2_d"], fl.FL_SIGMOID, True,
                small["sw13_d"], small["sw2_d"])[0].clone()
    b = run_moe(xb, logits, 3, small["I"], small["w13_d"], small["w2_d"], fl.FL_SIGMOID, True,
                small["sw13_d"], small["sw2_d"])[0].clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ------------------------------------------------------------------ full sizes

class DeviceExperts:
    """Expert weights drawn on the device (seeded), quantized and repacked on
    the device; fp32 weights of any expert can be redrawn for the oracle."""

    def __init__(self, E, H, I, layer, shared):
        self.E, self.H, self.I, self.layer = E, H, I, layer
        self.w13 = torch.cat([self._packed(e, 0) for e in range(E)])
        self.w2 = torch.cat([self._packed(e, 1) for e in range(E)])
        self.sw13 = self._packed(E, 0) if shared else None
        self.sw2 = self._packed(E, 1) if shared else None

    def fp32(self, e, which):
        N, K = (2 * self.I, self.H) if which == 0 else (self.H, self.I)
        return inputs.device_normal((N, K), 1, self.layer, e, which, device=DEV)

    def _packed(self, e, which):
        W = self.fp32(e, which)
        N, K = W.shape
        q, s, z = fl.fl_int4g_quantize(W)
        return fl.fl_int4g_repack(q, s, z, N, K)

    def oracle_triples(self, e, which):
        return O.quantize(self.fp32(e, which).cpu().numpy())


class LazyTriples:
    def __init__(self, ex, which):
        self.ex, self.which, self.cache = ex, which, {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = self.ex.oracle_triples(e, self.which)
        return self.cache[e]


def sampled_check(ex, xb, logits, k, scoring, y, ids, sample):
    w13 = LazyTriples(ex, 0)
    w2 = LazyTriples(ex, 1)
    # the oracle quantizes every expert the sampled tokens reach, in parallel
    need = sorted(set(ids.cpu().numpy()[sample].reshape(-1).tolist()))
    from oracle_pool import quantize_many
    jobs = [(e, which) for e in need for which in (0, 1)]
    if ex.sw13 is not None:
        jobs += [(ex.E, 0), (ex.E, 1)]
    trips = quantize_many(lambda i: ex.fp32(*jobs[i]).cpu().numpy(), len(jobs))
    for (e, which), t in zip(jobs, trips):
        (w13 if which == 0 else w2).cache[e] = t
    sw13 = w13.cache[ex.E] if ex.sw13 is not None else None
    sw2 = w2.cache[ex.E] if ex.sw2 is not None else None
    ref, tol, rid, _ = O.moe(O.bf16_value(xb[sample]), logits[sample], k, w13, w2, scoring, True, sw13, sw2)
    assert np.array_equal(ids.cpu().numpy()[sample], rid)
    check_y(y, ref, tol, rows=sample)


def covering_sample(ids, hot, extra=()):
    """Tokens to check at full size: greedily, until every expert of `hot`
    that received a token is covered; plus a token of the first and of the
    last routed expert (the first and last segments of the grouped kernels),
    the first and the last token, and `extra`."""
    ids = np.asarray(ids)
    M = ids.shape[0]
    want = set(int(e) for e in hot) & set(ids.reshape(-1).tolist())
    chosen = [0, M - 1]
    lo, hi = int(ids.min()), int(ids.max())
    chosen.append(int(np.nonzero((ids == lo).any(axis=1))[0][0]))
    chosen.append(int(np.nonzero((ids == hi).any(axis=1))[0][-1]))
    chosen += list(extra)
    for t in chosen:
        want -= set(ids[t].tolist())
    while want:
        gain = np.array([len(want & set(row.tolist())) for row in ids])
        t = int(np.argmax(gain))
        chosen.append(t)
        want -= set(ids[t].tolist())
    return np.unique(chosen)


def test_moe_qwen3_shaped():
    """128 experts, hidden 2048, intermediate 768, top-8 softmax; M in {1, 64,
    256} (M = 256 runs the grouped tensor-memory GEMM).  Sampled tokens: the
    first and last, a token of the first and of the last routed expert, and
    16 more spread over the batch."""
    ex = DeviceExperts(128, 2048, 768, layer=700, shared=False)
    for M in (1, 64, 256):
        xb = inputs.activations(M, 2048, stream=700 + M)
        logits = inputs.router_logits(M, 128, stream=700 + M)
        y, ids, wts, offs, perm = run_moe(xb, logits, 8, 768, ex.w13, ex.w2, fl.FL_SOFTMAX, True)
        check_routing(logits, 8, fl.FL_SOFTMAX, True, ids, wts, offs, perm)
        spread = np.linspace(0, M - 1, 16).astype(int) if M > 16 else np.arange(M)
        sample = covering_sample(ids.cpu().numpy(), [], extra=spread)
        sampled_check(ex, xb, logits, 8, O.SOFTMAX, y, ids, sample)


@pytest.mark.parametrize("M", [1, 16, 128, 512, 1024])
def test_moe_deepseek_shaped(M, deepseek_experts):
    """256 routed experts + 1 shared, hidden 7168, intermediate 2048, top-8
    sigmoid renormalised, logits skewed to 51 hot experts; M in {1, 16, 128,
    512, 1024} (M >= 128 runs the grouped tensor-memory GEMM).  Sampled
    tokens: every hot expert that received a token is covered by at least
    one of them, plus the first and last token and a token of the first and
    of the last routed expert (the grouped kernels' first and last
    segments; the shared expert's segments hold every token)."""
    ex = deepseek_experts
    xb = inputs.activations(M, 7168, stream=800 + M)
    logits = inputs.router_logits(M, 256, stream=800 + M, hot=51)
    y, ids, wts, offs, perm = run_moe(xb, logits, 8, 2048, ex.w13, ex.w2, fl.FL_SIGMOID, True, ex.sw13, ex.sw2)
    check_routing(logits, 8, fl.FL_SIGMOID, True, ids, wts, offs, perm)
    sample = covering_sample(ids.cpu().numpy(), inputs.hot_experts(256, 51))
    sampled_check(ex, xb, logits, 8, O.SIGMOID, y, ids, sample)


@pytest.fixture(scope="module")
def deepseek_experts():
    ex = DeviceExperts(256, 7168, 2048, layer=800, shared=True)
    yield ex
    del ex
    torch.cuda.empty_cache()


def test_moe_nan_logit_is_reported():
    """A NaN router logit is a device-side check failure (FL_ERR_DEVICE_CHECK
    in the status block); the NaN expert counts as -inf, so the routing of
    that token still picks valid experts and nothing is read out of bounds."""
    E, H, I, k, M = 8, 256, 128, 2, 4
    w13, w2 = host_experts(E, H, I, layer=96)
    xb = inputs.activations(M, H, stream=96)
    logits = inputs.router_logits(M, E, stream=96)
    logits[2, 5] = np.nan
    ids = torch.empty((M, k), dtype=torch.int32, device=DEV)
    ws = torch.zeros(fl.fl_moe_int4g_workspace(M, E, k, H, I, False), dtype=torch.uint8, device=DEV)
    fl.fl_moe_int4g(bf16_dev(xb), to_dev(logits), k, I, stack_dev(w13, 2 * I, H), stack_dev(w2, H, I),
                    topk_ids=ids, ws=ws)
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 6
    got = ids.cpu().numpy()
    assert np.all((got >= 0) & (got < E)) and 5 not in got[2].tolist()
    clean = logits.copy()
    clean[2, 5] = -np.inf
    rid, _ = O.route(clean, k, O.SOFTMAX, True)
    assert np.array_equal(got, rid)
    # the same workspace serves a clean call afterwards
    logits[2, 5] = 0.0
    y, ids, wts, offs, perm = run_moe(xb, logits, k, I, stack_dev(w13, 2 * I, H), stack_dev(w2, H, I),
                                      fl.FL_SOFTMAX, True)
    ref, tol, _, _ = O.moe(O.bf16_value(xb), logits, k, w13, w2, O.SOFTMAX, True)
    check_y(y, ref, tol)


@pytest.mark.parametrize("M", [5, 64])
def test_moe_group256_experts(M):
    """Experts quantized in groups of 256 (FastLLM page, section 4.2): the
    interleaved layout carries each group's scale in both of its 128-column
    super-blocks, and the MoE path (rows kernels at M=5, the grouped GEMM at
    M=64) runs on it unchanged."""
    E, H, I, k = 4, 512, 256, 2
    w13 = [O.quantize(inputs.expert_weight(2 * I, H, 97, e, 0), 256) for e in range(E)]
    w2 = [O.quantize(inputs.expert_weight(H, I, 97, e, 1), 256) for e in range(E)]
    w13_d = torch.cat([fl.fl_int4g_repack(to_dev(Q), to_dev(S.view(np.int16)), to_dev(Z), 2 * I, H, group=256)
                       for Q, S, Z in w13])
    w2_d = torch.cat([fl.fl_int4g_repack(to_dev(Q), to_dev(S.view(np.int16)), to_dev(Z), H, I, group=256)
                      for Q, S, Z in w2])
    xb = inputs.activations(M, H, stream=97)
    logits = inputs.router_logits(M, E, stream=97)
    y, ids, wts, offs, perm = run_moe(xb, logits, k, I, w13_d, w2_d, O.SOFTMAX, True)
    ref, tol, rid, rw = O.moe(O.bf16_value(xb), logits, k, w13, w2, O.SOFTMAX, True, group=256)
    assert np.array_equal(ids.cpu().numpy(), rid)
    check_y(y, ref, tol)


@pytest.mark.parametrize("M", [5, 64])
def test_moe_group64_experts(M):
    """Experts quantized in groups of 64 (FastLLM page, section 5.4): each
    expert matrix carries its side array; the rows kernels (M=5) and the
    grouped GEMM (M=64) read each 64-column group's scale and zero point.
    With a shared expert."""
    E, H, I, k = 4, 512, 256, 2
    w13 = [O.quantize(inputs.expert_weight(2 * I, H, 92, e, 0), 64) for e in range(E + 1)]
    w2 = [O.quantize(inputs.expert_weight(H, I, 92, e, 1), 64) for e in range(E + 1)]
    rp = lambda t, n, kk: fl.fl_int4g_repack(to_dev(t[0]), to_dev(t[1].view(np.int16)), to_dev(t[2]), n, kk, group=64)
    w13_d = torch.cat([rp(t, 2 * I, H) for t in w13[:E]])
    w2_d = torch.cat([rp(t, H, I) for t in w2[:E]])
    xb = inputs.activations(M, H, stream=92)
    logits = inputs.router_logits(M, E, stream=92)
    ids = torch.empty((M, k), dtype=torch.int32, device=DEV)
    ws = torch.zeros(fl.fl_moe_int4g_workspace(M, E, k, H, I, True), dtype=torch.uint8, device=DEV)
    y = fl.fl_moe_int4g(bf16_dev(xb), to_dev(logits), k, I, w13_d, w2_d, scoring=fl.FL_SIGMOID,
                        shared_w13=rp(w13[E], 2 * I, H), shared_w2=rp(w2[E], H, I), topk_ids=ids, ws=ws, group=64)
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 0
    ref, tol, rid, rw = O.moe(O.bf16_value(xb), logits, k, w13[:E], w2[:E], O.SIGMOID, True, w13[E], w2[E],
                              group=64)
    assert np.array_equal(ids.cpu().numpy(), rid)
    check_y(y, ref, tol)


def _routing_case(M, E, k, H, I, layer):
    w13, w2 = host_experts(E, H, I, layer)
    w13_d, w2_d = stack_dev(w13, 2 * I, H), stack_dev(w2, H, I)
    xb = inputs.activations(M, H, stream=layer)
    logits = inputs.router_logits(M, E, stream=layer, hot=max(1, E // 5))
    return w13, w2, w13_d, w2_d, xb, logits


def _run_moe_ex(xb, logits, k, I, w13_d, w2_d, scoring, **opts):
    M, H = xb.shape
    E = logits.shape[1]
    ids = torch.empty((M, k), dtype=torch.int32, device=DEV)
    wts = torch.empty((M, k), dtype=torch.float32, device=DEV)
    ws = torch.zeros(fl.fl_moe_int4g_workspace(M, E, k, H, I, False), dtype=torch.uint8, device=DEV)
    if opts.get("score_bias") is not None:
        opts = dict(opts, score_bias=to_dev(opts["score_bias"]))
    y = fl.fl_moe_int4g(bf16_dev(xb), to_dev(logits), k, I, w13_d, w2_d, scoring=scoring, renorm=True,
                        topk_ids=ids, topk_w=wts, ws=ws, **opts)
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 0
    return y, ids, wts


@pytest.mark.parametrize("opts", [
    {"n_group": 8, "topk_group": 4},
    {"bias": True},
    {"bias": True, "n_group": 8, "topk_group": 4, "routed_scale": 2.5},
])
def test_moe_deepseek_routing_options(opts):
    """Sigmoid affinities with the selection bias, group-limited top-k (8
    groups of 32, 4 kept) and the routed scale, on 256 small experts: ids
    bit-exact (keys compared in double on both sides), weights within 1e-5
    relative, y within the propagated bound."""
    M, E, k, H, I = 96, 256, 8, 256, 128
    w13, w2, w13_d, w2_d, xb, logits = _routing_case(M, E, k, H, I, layer=98)
    ro = {"n_group": opts.get("n_group", 1), "topk_group": opts.get("topk_group", 1),
          "scale": opts.get("routed_scale", 1.0)}
    dev_opts = {"n_group": ro["n_group"], "topk_group": ro["topk_group"], "routed_scale": ro["scale"]}
    if opts.get("bias"):
        bias = (0.05 * np.random.default_rng([0, 6, 98]).standard_normal(E)).astype(np.float32)
        ro["bias"] = bias
        dev_opts["score_bias"] = bias
    y, ids, wts = _run_moe_ex(xb, logits, k, I, w13_d, w2_d, O.SIGMOID, **dev_opts)
    ref, tol, rid, rw = O.moe(O.bf16_value(xb), logits, k, w13, w2, O.SIGMOID, True, routing=ro)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(wts.cpu().numpy(), rw, rtol=1e-5, atol=0)
    check_y(y, ref, tol)


def test_moe_routed_scale_softmax():
    M, E, k, H, I = 9, 8, 2, 256, 128
    w13, w2, w13_d, w2_d, xb, logits = _routing_case(M, E, k, H, I, layer=99)
    y, ids, wts = _run_moe_ex(xb, logits, k, I, w13_d, w2_d, O.SOFTMAX, routed_scale=2.5)
    ref, tol, rid, rw = O.moe(O.bf16_value(xb), logits, k, w13, w2, O.SOFTMAX, True, routing={"scale": 2.5})
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.allclose(wts.cpu().numpy(), rw, rtol=1e-5, atol=0)
    check_y(y, ref, tol)


@pytest.mark.parametrize("M", [5, 96])
def test_moe_expert_pointer_tables(M):
    """Experts in separate allocations, passed as device tables of pointers
    (fl_moe_int4g_ptrs): the same bits as the back-to-back call, on the rows
    kernels (M = 5) and the grouped GEMM (M = 96, 24 positions per expert)."""
    E, H, I, k = 8, 512, 256, 2
    w13, w2 = host_experts(E, H, I, layer=95)
    sw13, sw2 = host_experts(1, H, I, layer=94)
    w13_each = [repack_dev(*t, 2 * I, H) for t in w13]
    w2_each = [repack_dev(*t, H, I) for t in w2]
    xb = inputs.activations(M, H, stream=95)
    logits = inputs.router_logits(M, E, stream=95)
    sd13, sd2 = repack_dev(*sw13[0], 2 * I, H), repack_dev(*sw2[0], H, I)
    y_ref, ids, wts, offs, perm = run_moe(xb, logits, k, I, torch.cat(w13_each), torch.cat(w2_each), fl.FL_SIGMOID,
                                          True, sd13, sd2)
    y_ref = y_ref.clone()
    ws = torch.zeros(fl.fl_moe_int4g_workspace(M, E, k, H, I, True), dtype=torch.uint8, device=DEV)
    y = fl.fl_moe_int4g_ptrs(bf16_dev(xb), to_dev(logits), k, I, w13_each, w2_each, scoring=fl.FL_SIGMOID,
                             shared_w13=sd13, shared_w2=sd2, ws=ws)
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 0
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16))
    ref, tol, _, _ = O.moe(O.bf16_value(xb), logits, k, w13, w2, O.SIGMOID, True, sw13[0], sw2[0])
    check_y(y, ref, tol)


def test_moe_expert_pointer_table_bad_entry_is_reported():
    """A misaligned table entry is caught on the device (FL_ERR_DEVICE_CHECK):
    that expert's copies are skipped (no fault), the call completes."""
    E, H, I, k, M = 4, 256, 128, 2, 6
    w13, w2 = host_experts(E, H, I, layer=93)
    w13_each = [repack_dev(*t, 2 * I, H) for t in w13]
    w2_each = [repack_dev(*t, H, I) for t in w2]
    xb = inputs.activations(M, H, stream=93)
    logits = inputs.router_logits(M, E, stream=93)
    logits[:, 1] += 10.0   # every token is routed to expert 1
    t13 = torch.tensor([t.data_ptr() for t in w13_each], dtype=torch.int64, device=DEV)
    t2 = torch.tensor([t.data_ptr() for t in w2_each], dtype=torch.int64, device=DEV)
    t13[1] += 8   # misaligned: 8 bytes past expert 1's start (inside its buffer)
    ws = torch.zeros(fl.fl_moe_int4g_workspace(M, E, k, H, I, False), dtype=torch.uint8, device=DEV)
    fl.fl_moe_int4g_ptrs(bf16_dev(xb), to_dev(logits), k, I, w13_each, w2_each, ws=ws, tables=(t13, t2))
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 6


# ------------------------------------------------------------------ router projection

def _router_case(M, H, E, layer):
    rng = np.random.default_rng([0, 7, layer])
    w = inputs.to_bf16_bits((rng.standard_normal((E, H)) * 0.02).astype(np.float32))
    xb = inputs.activations(M, H, stream=layer)
    return xb, w


@pytest.mark.parametrize("MHE", [(1, 7168, 256), (16, 7168, 256), (128, 7168, 256), (1024, 7168, 256),
                                 (1, 2048, 128), (256, 2048, 128), (37, 192, 70), (130, 256, 8)])
def test_router_logits_parity(MHE):
    """Router logits against the oracle's double projection, every output,
    within 2e-3 * sum |x||Wr| + 1e-5; two calls give the same bits (the
    split-K partials are added in a fixed order)."""
    M, H, E = MHE
    xb, wb = _router_case(M, H, E, layer=M + H + E)
    x = bf16_dev(xb)
    w = bf16_dev(wb)
    ws = torch.zeros(fl.fl_moe_router_logits_workspace(M, H, E), dtype=torch.uint8, device=DEV)
    l1 = fl.fl_moe_router_logits(x, w, ws=ws).clone()
    l2 = fl.fl_moe_router_logits(x, w, ws=ws).clone()
    torch.cuda.synchronize()
    assert torch.equal(l1, l2)
    ref, tol = O.router_logits(O.bf16_value(xb), O.bf16_value(wb))
    got = l1.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= tol), np.max(np.abs(got - ref) / tol)


def test_router_then_moe_deepseek_routing():
    """The router projection feeding the layer (DeepSeek-V3-shaped router:
    H=7168, E=256, top-8 sigmoid): the ids chosen from the device logits
    equal the oracle's wherever the oracle's k-th and (k+1)-th logits are
    further apart than the logits' error bound; elsewhere either choice is
    correct and the chosen experts must be among the near-tied ones."""
    M, H, E, k = 64, 7168, 256, 8
    xb, wb = _router_case(M, H, E, layer=77)
    logits = fl.fl_moe_router_logits(bf16_dev(xb), bf16_dev(wb))
    torch.cuda.synchronize()
    ref, tol = O.router_logits(O.bf16_value(xb), O.bf16_value(wb))
    # routing of the device logits on the device (small experts: only the ids matter here)
    Ie, He = 128, H
    ids = torch.empty((M, k), dtype=torch.int32, device=DEV)
    ex13 = torch.zeros(fl.fl_int4g_repacked_bytes(2 * Ie, He) * E, dtype=torch.uint8, device=DEV)
    ex2 = torch.zeros(fl.fl_int4g_repacked_bytes(He, Ie) * E, dtype=torch.uint8, device=DEV)
    fl.fl_moe_int4g(bf16_dev(xb), logits, k, Ie, ex13, ex2, scoring=fl.FL_SIGMOID, topk_ids=ids)
    torch.cuda.synchronize()
    got = ids.cpu().numpy()
    rid, _ = O.route(ref.astype(np.float32), k, O.SIGMOID, True)
    for t in range(M):
        order = np.sort(ref[t])[::-1]
        margin = order[k - 1] - order[k]
        if margin > 2 * tol[t].max():
            assert set(got[t].tolist()) == set(rid[t].tolist()), t
        else:
            assert np.all(ref[t][got[t]] >= order[k - 1] - 2 * tol[t].max()), t
