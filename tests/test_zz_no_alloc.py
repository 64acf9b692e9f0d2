"""The decode linear variant that allocates nothing (fl_int4g_linear_noalloc),
for callers that cannot allocate device memory where they call, against the
workspace entry point (fl_int4g_linear, bit for bit: both run the same
kernels) and against the CPU oracle (elementwise bound), two calls in a row.
Collected last: it shares a library-wide scratch array."""
import ctypes

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


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def _case(M, N, K, layer):
    W = inputs.dense_weight(N, K, layer=layer)
    q, s, z = fl.fl_int4g_quantize(_dev(W))
    w = fl.fl_int4g_repack(q, s, z, N, K)
    xb = inputs.activations(M, K, stream=layer)
    return W, w, xb, _dev(xb.view(np.int16)).view(torch.bfloat16)


def _oracle_cols(W, xb, cols):
    Qr, Sr, Zr = O.quantize(W[cols])
    return O.linear_columns(O.bf16_value(xb), Qr, Sr, Zr, np.arange(len(cols)))


# M = 1..8: the mma.sync decode kernel; 12, 24, 32: the tcgen05 decode kernel
@pytest.mark.parametrize("M", [1, 5, 8, 12, 24, 32])
@pytest.mark.parametrize("NK", [(200, 384), (512, 1280)])
def test_noalloc_small_every_output(M, NK):
    N, K = NK
    W, w, xb, x = _case(M, N, K, layer=980 + M + K)
    y_ws = fl.fl_int4g_linear(x, w, N).clone()
    ref, tol = _oracle_cols(W, xb, np.arange(N))
    for _ in range(2):
        y = fl.fl_int4g_linear_noalloc(x, w, N)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_ws.view(torch.int16))
        got = y.float().cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= tol), np.max(np.abs(got - ref) / tol)
    assert fl.fl_int4g_linear_noalloc_status() == 0


@pytest.mark.parametrize("MNK", [(1, 3072, 1024), (8, 12288, 4096), (12, 11008, 4096), (32, 4096, 11008)])
def test_noalloc_full_size_sampled(MNK):
    M, N, K = MNK
    W, w, xb, x = _case(M, N, K, layer=990 + M)
    y_ws = fl.fl_int4g_linear(x, w, N).clone()
    cols = np.unique(np.concatenate([np.linspace(0, N - 1, 64).astype(int), [N - 1]]))
    ref, tol = _oracle_cols(W, xb, cols)
    for _ in range(2):
        y = fl.fl_int4g_linear_noalloc(x, w, N)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), y_ws.view(torch.int16))
        got = y.float().cpu().numpy().astype(np.float64)[:, cols]
        assert np.all(np.abs(got - ref) <= tol), np.max(np.abs(got - ref) / tol)
    assert fl.fl_int4g_linear_noalloc_status() == 0


def test_noalloc_rejects_beyond_its_scratch():
    L = fl.lib()
    fake = ctypes.c_void_p(0x10000)
    # M > 32 is not a decode shape; a very tall N at M = 32 needs more scratch than the array holds
    assert L.fl_int4g_linear_noalloc(fake, 33, 256, fake, 128, fake, None) == 3
    assert L.fl_int4g_linear_noalloc(fake, 32, 256, fake, 1000000, fake, None) == 2
