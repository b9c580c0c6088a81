"""Failure detection without a GPU fault: the stochastic sampler's bounded wait runs out
on a sequence whose decision nothing publishes (spec_selftest_wait_timeout: no tile
kernel runs, so neither the record nor the tile count ever completes). The kernel
reports SPEC_DEV_TIMEOUT and returns, and the context stays usable."""
import ctypes
import time

import pytest
import torch

from speculative_decoding_token_temp_gb300 import _lib, synth

from gpu_util import compare_stochastic, handmade, run_stochastic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def test_bounded_wait_reports_timeout(dev):
    lib = _lib.lib()
    g = _lib.SpecBatch(1, 1, 8, 1, None)
    nbytes = lib.spec_workspace_bytes(g, _lib.SPEC_BF16, _lib.SPEC_MODE_STOCHASTIC)
    ws = torch.full((nbytes,), 0xA5, dtype=torch.uint8, device=dev)   # stale contents: the prologue re-arms
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    P = ctypes.c_void_p
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    code = lib.spec_selftest_wait_timeout(P(status.data_ptr()), P(ws.data_ptr()), ws.numel(), P(stream))
    assert code == _lib.SPEC_OK
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert int(status.item()) == _lib.SPEC_DEV_TIMEOUT
    assert waited < 5.0, waited
    print(f"bounded wait gave up after {waited * 1e3:.0f} ms")
    # the context is usable: an ordinary call on the same stream
    w = handmade(3, 4, 2048, synth.BF16, T=0.8, seed=99)
    res = run_stochastic(w, dev)
    assert res["device_status"][0] == 0
    compare_stochastic(w, res, range(w.B))
