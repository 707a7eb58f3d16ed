"""q8_1 quantiser on the GPU: bit-exact against the oracle (quants, d, s)."""
import numpy as np
import pytest

import synth
from helpers import ensure_lib, to_np
from oracle import q8_1 as oq

pytestmark = pytest.mark.gpu


def _edge_rows(K):
    """Rows with a zero block, a 3e4 outlier, exact half ties and negative amax."""
    rows = []
    z = np.zeros(K, np.float32)
    rows.append(z)
    o = synth.activations(synth.rng(1), 1, K)[0]
    o[3] = 3e4
    rows.append(o)
    t = np.zeros(K, np.float32)
    t[0], t[1], t[2], t[3] = 127, 2.5, -2.5, 0.5        # d = 1, ties away from zero
    rows.append(t)
    n = np.zeros(K, np.float32)
    n[0], n[1] = -0.5, 0.25                             # division lands exactly on 63.5
    rows.append(n)
    tiny = synth.activations(synth.rng(2), 1, K)[0] * 1e-30   # subnormal-range d
    rows.append(tiny)
    return np.stack(rows).astype(np.float32)


@pytest.mark.parametrize("ncols,K", [(1, 32), (3, 2560), (8, 2048), (11, 96), (64, 64), (5, 1536)])
def test_quantize_bit_exact(ncols, K):
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    x = synth.activations(synth.rng(100 + K), ncols, K) * 3
    if ncols >= 5:
        x[-5:] = _edge_rows(K)
    xt = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    q, ds = mx.quantize_q8_1(xt)
    torch.cuda.synchronize()
    rq, rd, rs = oq.quantize_q8_1(x)
    assert np.array_equal(to_np(q), rq)
    g = to_np(ds)
    assert np.array_equal(g[..., 0].view(np.uint32), rd.view(np.uint32))
    assert np.array_equal(g[..., 1].view(np.uint32), rs.view(np.uint32))
    assert mx.device_status() == 0


def test_quantize_strided_columns():
    import torch
    import moe_expert_gb300 as mx
    ensure_lib()
    K, ncols, ld = 2560, 4, 2560 + 64
    base = synth.activations(synth.rng(7), ncols, ld)
    xt = torch.from_numpy(base).cuda()
    q = torch.empty((ncols, K), dtype=torch.int8, device="cuda")
    ds = torch.empty((ncols, K // 32, 2), dtype=torch.float32, device="cuda")
    import ctypes
    st = mx.lib().moex_quantize_q8_1(ctypes.c_void_p(xt.data_ptr()), K, ncols, ld, ctypes.c_void_p(q.data_ptr()),
                                     ctypes.c_void_p(ds.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    rq, rd, rs = oq.quantize_q8_1(base[:, :K])
    assert np.array_equal(to_np(q), rq)
    assert np.array_equal(to_np(ds)[..., 0], rd)
