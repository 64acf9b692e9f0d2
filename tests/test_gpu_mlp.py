"""GPU parity of the fused decode MLP block (fl_int4g_mlp: gate/up, SwiGLU
and down in one launch) through the C ABI against the CPU oracle: the
oracle's expert FFN (h = silu(G x) * (U x) stored as bf16, y = D h) with its
propagated elementwise bound, widened by the bf16 store of y."""
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


def repack_dev(Q, S, Z, N, K):
    return fl.fl_int4g_repack(to_dev(Q), to_dev(S.view(np.int16)), to_dev(Z), N, K)


def mlp_case(H, I, layer):
    """Oracle-quantized gate, up and down of one MLP block, and their
    interleaved device copies."""
    G = O.quantize(inputs.dense_weight(I, H, layer=layer))
    U = O.quantize(inputs.dense_weight(I, H, layer=layer + 1))
    D = O.quantize(inputs.dense_weight(H, I, layer=layer + 2))
    dev = (repack_dev(*G, I, H), repack_dev(*U, I, H), repack_dev(*D, H, I))
    return G, U, D, dev


def oracle_mlp(xb, G, U, D):
    """The oracle's MoE layer with one expert and weight 1 is exactly the
    MLP block: W13 = [G; U] (gate rows first), W2 = D."""
    w13 = tuple(np.concatenate([a, b], axis=0) for a, b in zip(G, U))
    M = xb.shape[0]
    y, tol, _, _ = O.moe(O.bf16_value(xb), np.zeros((M, 1), np.float32), 1, [w13], [D], O.SOFTMAX, True)
    return y, tol


def check(y, ref, tol):
    got = y.float().cpu().numpy().astype(np.float64)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= tol), f"worst err/tol {np.max(err / tol):.3f} at {np.unravel_index(np.argmax(err / tol), err.shape)}"
    rel = np.sqrt(np.mean(err ** 2) / np.mean(ref ** 2))
    assert rel <= 1e-2, f"relative RMS error {rel:.3e}"


@pytest.mark.parametrize("one_launch", [False, True])
@pytest.mark.parametrize("M", [1, 3, 8])
@pytest.mark.parametrize("HI", [(256, 256), (384, 640), (1024, 384), (128, 128), (4096, 1408)])
def test_mlp_small_every_output(M, HI, one_launch):
    H, I = HI
    G, U, D, (g, u, d) = mlp_case(H, I, layer=1200 + H + I)
    xb = inputs.activations(M, H, stream=1200 + M)
    ws = torch.zeros(fl.fl_int4g_mlp_workspace(M, H, I), dtype=torch.uint8, device=DEV)
    x = to_dev(xb.view(np.int16)).view(torch.bfloat16)
    y = fl.fl_int4g_mlp(x, g, u, d, I, ws=ws, one_launch=one_launch)
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 0
    ref, tol = oracle_mlp(xb, G, U, D)
    check(y, ref, tol)


@pytest.mark.parametrize("one_launch", [False, True])
@pytest.mark.parametrize("M", [1, 8])
def test_mlp_llama_full(M, one_launch):
    """Llama-7B MLP block (H=4096, I=11008) at M in {1, 8}, every output;
    two calls on one workspace give the same bits (the counters are left
    zero, the reduction order is fixed)."""
    H, I = 4096, 11008
    G, U, D, (g, u, d) = mlp_case(H, I, layer=1300)
    xb = inputs.activations(M, H, stream=1300 + M)
    x = to_dev(xb.view(np.int16)).view(torch.bfloat16)
    ws = torch.zeros(fl.fl_int4g_mlp_workspace(M, H, I), dtype=torch.uint8, device=DEV)
    y1 = fl.fl_int4g_mlp(x, g, u, d, I, ws=ws, one_launch=one_launch).clone()
    y2 = fl.fl_int4g_mlp(x, g, u, d, I, ws=ws, one_launch=one_launch).clone()
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 0
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    ref, tol = oracle_mlp(xb, G, U, D)
    check(y1, ref, tol)


@pytest.mark.parametrize("M", [1, 8])
def test_mlp_long_hidden(M):
    """H=16384, I=256: the gate/up half runs in clusters of 8 ranks of 16
    groups.  At M=1 each rank keeps the x rows of its slice in an x region of
    shared memory; at M=8 that region would leave fewer than three stages,
    so x travels in the stages.  Every output against the oracle."""
    H, I = 16384, 256
    G, U, D, (g, u, d) = mlp_case(H, I, layer=1600)
    xb = inputs.activations(M, H, stream=1600 + M)
    ws = torch.zeros(fl.fl_int4g_mlp_workspace(M, H, I), dtype=torch.uint8, device=DEV)
    x = to_dev(xb.view(np.int16)).view(torch.bfloat16)
    y = fl.fl_int4g_mlp(x, g, u, d, I, ws=ws)
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 0
    ref, tol = oracle_mlp(xb, G, U, D)
    check(y, ref, tol)


@pytest.mark.parametrize("one_launch", [False, True])
def test_mlp_in_a_cuda_graph(one_launch):
    """Both forms (the cooperative launch among them) captured in a CUDA
    graph and replayed."""
    M, H, I = 2, 512, 384
    G, U, D, (g, u, d) = mlp_case(H, I, layer=1400)
    xb = inputs.activations(M, H, stream=1400)
    x = to_dev(xb.view(np.int16)).view(torch.bfloat16)
    ws = torch.zeros(fl.fl_int4g_mlp_workspace(M, H, I), dtype=torch.uint8, device=DEV)
    y = torch.empty((M, H), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        fl.fl_int4g_mlp(x, g, u, d, I, y=y, ws=ws, one_launch=one_launch)
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        fl.fl_int4g_mlp(x, g, u, d, I, y=y, ws=ws, one_launch=one_launch)
    y.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 0
    ref, tol = oracle_mlp(xb, G, U, D)
    check(y, ref, tol)


def test_mlp_rejects_bad_arguments():
    import ctypes
    L = fl.lib()
    fake = ctypes.c_void_p(0x10000)
    assert L.fl_int4g_mlp(fake, 9, 256, 256, fake, fake, fake, fake, fake, 1 << 30, None) == 3   # M > 8
    assert L.fl_int4g_mlp_fused(fake, 9, 256, 256, fake, fake, fake, fake, fake, 1 << 30, None) == 3
    assert L.fl_int4g_mlp(fake, 1, 200, 256, fake, fake, fake, fake, fake, 1 << 30, None) == 1   # H % 128
    assert L.fl_int4g_mlp(fake, 1, 256, 256, fake, fake, fake, fake, fake, 16, None) == 2        # workspace


def test_mlp_glu_timeout_is_reported():
    """The gate/up launch reduces row tiles across thread-block clusters: the
    test hook makes that bounded wait run out (FL_ERR_TIMEOUT reported, no
    hang, no fault), and the next call on the workspace is correct."""
    M, H, I = 2, 512, 256
    G, U, D, (g, u, d) = mlp_case(H, I, layer=1500)
    xb = inputs.activations(M, H, stream=1500)
    x = to_dev(xb.view(np.int16)).view(torch.bfloat16)
    ws = torch.zeros(fl.fl_int4g_mlp_workspace(M, H, I), dtype=torch.uint8, device=DEV)
    fl.fl_int4g_test_withhold_cluster_arrival(1_000_000)
    try:
        fl.fl_int4g_mlp(x, g, u, d, I, ws=ws)
        torch.cuda.synchronize()
    finally:
        fl.fl_int4g_test_withhold_cluster_arrival(-1)
    assert fl.fl_int4g_status(ws) == 5
    y = fl.fl_int4g_mlp(x, g, u, d, I, ws=ws)
    torch.cuda.synchronize()
    assert fl.fl_int4g_status(ws) == 0
    ref, tol = oracle_mlp(xb, G, U, D)
    check(y, ref, tol)
