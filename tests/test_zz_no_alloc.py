"""kamera_factor_patches_noalloc: patch formation for callers that cannot
allocate device memory -- for example a serving engine that owns all device
memory through its own allocator, or a plugin hook whose enqueue step must
not allocate (cudaMalloc / cudaFree can synchronise the device).  Its scratch
is a fixed static array inside the library instead of a caller workspace.

It must give the same factors as kamera_factor_patches with a workspace, on
consecutive calls (the array keeps the previous call's contents, which must
not leak into the next result).  The comparison is bit for bit, which is
within every tolerance the other tests use.  This file is collected last so
that a failure here stops a -x run only after everything else has run.
"""
import numpy as np
import pytest

from synth import gen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _run_both(deltas: np.ndarray, m: int, p: int, q: int, seed: int):
    import position_invariant_kv_kamera_gb300 as pk

    n, T, D = deltas.shape
    d_dev = torch.from_numpy(np.ascontiguousarray(deltas)).cuda()
    om = torch.from_numpy(gen.gaussian_test_matrix(seed, D, m + p)).cuda()
    desc = pk.factor_desc(d_dev, n, T, D, m, p, q, om)
    stride = (T + D) * m
    stream = pk.stream_handle()
    # the existing entry point, with a workspace the caller allocates
    nbytes = pk.kamera_factor_workspace_size(desc)
    ws = torch.empty(nbytes // 4 + 64, dtype=torch.float32, device="cuda")
    out_ws = torch.full((n * stride,), -1, dtype=torch.int16, device="cuda")
    pk.kamera_factor_patches(desc, out_ws.data_ptr(), out_ws.data_ptr() + 2 * T * m, stride, ws.data_ptr(), nbytes,
                             stream)
    # the allocation-free entry point, through the C ABI
    out_static = torch.full((n * stride,), -1, dtype=torch.int16, device="cuda")
    pk.kamera_factor_patches_noalloc(desc, out_static.data_ptr(), out_static.data_ptr() + 2 * T * m, stride, stream)
    torch.cuda.synchronize()
    return out_ws.cpu().numpy().view(np.uint16), out_static.cpu().numpy().view(np.uint16)


def test_noalloc_matches_workspace_entry_point_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    # call 1: 60 slabs of 1024 x 512 -- more than the static scratch can serve
    # at once (it runs on fewer CTAs, each taking several slabs)
    d1 = np.stack([gen.low_rank_deficit(31, s, 1024, 512, np.linspace(6, 1, 40)) for s in range(60)])
    a1, b1 = _run_both(d1, m=32, p=16, q=2, seed=7)
    assert (a1 != 0xFFFF).all()
    np.testing.assert_array_equal(b1, a1)
    # call 2: another shape and rank; whatever call 1 left in the array must not matter
    d2 = np.stack([gen.low_rank_deficit(32, s, 300, 256, np.linspace(9, 2, 12), noise=1e-3) for s in range(5)])
    a2, b2 = _run_both(d2, m=16, p=16, q=1, seed=8)
    assert (a2 != 0xFFFF).all()
    np.testing.assert_array_equal(b2, a2)
