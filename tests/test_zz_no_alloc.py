"""The decode linear variant that allocates nothing (fl_int4g_linear_noalloc),
for callers that cannot allocate device memory where they call, against the
workspace entry point (fl_int4g_linear) on the same inputs, two calls in a
row.  Collected last: it shares a library-wide scratch array."""
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


@pytest.mark.parametrize("MNK", [(1, 3072, 1024), (8, 12288, 4096), (32, 4096, 11008), (5, 200, 384)])
def test_noalloc_matches_workspace_entry_point(MNK):
    M, N, K = MNK
    W = inputs.dense_weight(N, K, layer=990 + M)
    q, s, z = fl.fl_int4g_quantize(_dev(W))
    w = fl.fl_int4g_repack(q, s, z, N, K)
    xb = inputs.activations(M, K, stream=990 + M)
    x = _dev(xb.view(np.int16)).view(torch.bfloat16)
    y_ws = fl.fl_int4g_linear(x, w, N).clone()
    # tolerance of the parity tests, from the oracle on a sample of rows
    rows = np.unique(np.linspace(0, N - 1, 64).astype(int))
    Qr, Sr, Zr = O.quantize(W[rows])
    _, tol = O.linear_columns(O.bf16_value(xb), Qr, Sr, Zr, np.arange(len(rows)))
    for _ in range(2):
        y = fl.fl_int4g_linear_noalloc(x, w, N)
        torch.cuda.synchronize()
        d = (y.float() - y_ws.float()).abs().cpu().numpy().astype(np.float64)
        assert np.all(d[:, rows] <= tol)
        assert np.all(d <= np.max(tol))


def test_noalloc_rejects_beyond_its_scratch():
    L = fl.lib()
    fake = ctypes.c_void_p(0x10000)
    # M > 32 is not a decode shape; a very tall N at M = 32 needs more scratch than the array holds
    assert L.fl_int4g_linear_noalloc(fake, 33, 256, fake, 128, fake, None) == 3
    assert L.fl_int4g_linear_noalloc(fake, 32, 256, fake, 1000000, fake, None) == 2
