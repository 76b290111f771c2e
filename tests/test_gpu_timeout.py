"""The expiry path of the kernel's bounded waits, made to run out without any
fault.  A test-only launch setting shortens the bound of every wait to 1 ms
and has each CTA's producer leave its first canonical stage unfilled with its
barrier unarmed.  The waits on that stage then give up: the kernel must set
KAMERA_EFLAG_TIMEOUT (and no other bit), stop, wait for its own copies and
tensor-core work in flight, release its tensor memory and return -- well
within a second -- and the same stream must then run a normal call whose
pool matches the oracle."""
import time

import numpy as np
import pytest

from synth import workloads as W
from tests import harness as H

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import position_invariant_kv_kamera_gb300 as pk  # noqa: E402

CASES = {
    # patched reuse from the store: TMA loads, tensor-core patch, TMA stores
    "reuse_patched": lambda: W.gqa_video(num_layers=2, n_chunks=3, T=300, rank=32, page_size=16),
    # in-place sliding-window relocation: no patch, no tensor memory
    "relocate_in_place": lambda: W.sliding_window(num_layers=2, n_resident=5, n_evict=1, T=256, page_size=64,
                                                  num_kv_heads=4),
}


@pytest.fixture(autouse=True)
def _cuda_and_default_tuning():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    pk.kamera_set_launch_tuning()
    yield
    pk.kamera_set_launch_tuning()


@pytest.mark.parametrize("name", sorted(CASES))
def test_wait_expiry_reports_timeout_and_the_stream_stays_usable(name):
    wl = CASES[name]()
    pool = (wl.host_pool(0), wl.host_pool(1) if wl.n_ch == 2 else None)
    t = H.device_inputs(wl, torch, pool_host=pool)
    torch.cuda.synchronize()

    pk.kamera_set_launch_tuning(wait_limit_ns=1_000_000, test_unarm_first_stage=1)
    t0 = time.perf_counter()
    try:
        assert H.call(wl, t) == pk.KAMERA_OK
        torch.cuda.synchronize()
    finally:
        pk.kamera_set_launch_tuning()
    elapsed = time.perf_counter() - t0
    err = int(t["err"].item())
    assert err & pk.KAMERA_EFLAG_TIMEOUT, err
    assert err & ~pk.KAMERA_EFLAG_TIMEOUT == 0, err
    assert elapsed < 1.0, elapsed  # the 1 ms bound held, not the 2 s default

    # the defaults are back (0 = the library's choice, a 2 s bound)
    tune = pk.kamera_get_launch_tuning()
    assert tune.wait_limit_ns == 0 and tune.test_unarm_first_stage == 0

    # a normal call on the same stream, from fresh inputs, matches the oracle
    t2 = H.device_inputs(wl, torch, pool_host=pool)
    H.call(wl, t2)
    torch.cuda.synchronize()
    assert int(t2["err"].item()) == 0
    err_ref, ref_k, ref_v, wk, wv = H.oracle_reference(wl, pool[0], pool[1])
    assert err_ref == 0
    H.assert_report(H.compare_pool(H.to_bits(t2["pool_k"]), pool[0], ref_k, wk))
    if wl.n_ch == 2:
        H.assert_report(H.compare_pool(H.to_bits(t2["pool_v"]), pool[1], ref_v, wv))
