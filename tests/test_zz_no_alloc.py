"""spec_verify_stochastic_static: stochastic verification for callers that cannot allocate.

Some callers only get the buffers a host framework hands them (a plugin whose memory
pool belongs to an inference server, a decode loop that must not call cudaMalloc or
cudaFree). This entry point takes no workspace: its scratch is a fixed array inside the
library. These tests call it through the C ABI and check that two calls in a row give
what the workspace-taking entry point gives on the same inputs, within the tolerances
of the other parity tests. The file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_token_temp_gb300 import _lib, api, synth

pytestmark = pytest.mark.gpu

REL = 1e-4
NKL_ABS = 2e-6


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _t(a, dev):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


def test_static_scratch_matches_workspace_call(dev):
    w = synth.MID.make(T=0.6)
    g = int(w.gammas[0])
    t, d = _t(w.target, dev), _t(w.draft, dev)
    tok, ua, us = _t(w.tokens, dev), _t(w.u_accept, dev), _t(w.u_sample, dev)
    ref = api.spec_verify_stochastic(t, d, tok, w.T, ua, us, gamma=g)
    torch.cuda.synchronize()
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    assert ref["device_status"][0] == 0

    lib = _lib.lib()
    batch = _lib.SpecBatch(w.B, g, w.V, w.total_draft, None)
    assert lib.spec_workspace_bytes(batch, _lib.SPEC_BF16, _lib.SPEC_MODE_STOCHASTIC) <= _lib.SPEC_STATIC_SCRATCH_BYTES
    P = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    rows, tot = w.total_target, w.total_draft
    for call in range(2):
        o = {"n_accepted": torch.full((w.B,), -7, dtype=torch.int32, device=dev),
             "out_tokens": torch.full((rows,), -7, dtype=torch.int32, device=dev),
             "p_x": torch.full((tot,), -7.0, device=dev), "q_x": torch.full((tot,), -7.0, device=dev),
             "alpha": torch.full((tot,), -7.0, device=dev), "nkl": torch.full((tot,), -7.0, device=dev),
             "nkl_mask": torch.full((tot,), 7, dtype=torch.uint8, device=dev),
             "greedy_n": torch.full((w.B,), -7, dtype=torch.int32, device=dev),
             "greedy_tokens": torch.full((rows,), -7, dtype=torch.int32, device=dev),
             "device_status": torch.zeros(1, dtype=torch.int32, device=dev)}
        code = lib.spec_verify_stochastic_static(
            batch, _lib.SPEC_BF16, P(t), P(d), P(tok), w.T, P(ua), P(us), P(o["n_accepted"]), P(o["out_tokens"]),
            P(o["p_x"]), P(o["q_x"]), P(o["alpha"]), P(o["nkl"]), P(o["nkl_mask"]), 0.15, P(o["greedy_n"]),
            P(o["greedy_tokens"]), P(o["device_status"]), stream)
        assert code == _lib.SPEC_OK, _lib.status_str(code)
        torch.cuda.synchronize()
        got = {k: v.cpu().numpy() for k, v in o.items()}
        assert got["device_status"][0] == 0, call
        for k in ("n_accepted", "out_tokens", "greedy_n", "greedy_tokens", "nkl_mask"):
            assert np.array_equal(got[k], ref[k]), (call, k)
        for k in ("p_x", "q_x", "alpha"):
            assert np.allclose(got[k], ref[k], rtol=REL, atol=0), (call, k)
        assert np.allclose(got["nkl"], ref["nkl"], rtol=REL, atol=NKL_ABS), call


def test_static_scratch_rejects_problems_beyond_its_size(dev):
    lib = _lib.lib()
    big = _lib.SpecBatch(4096, 16, 152064, 4096 * 16, None)
    assert lib.spec_workspace_bytes(big, _lib.SPEC_BF16, _lib.SPEC_MODE_STOCHASTIC) > _lib.SPEC_STATIC_SCRATCH_BYTES
    one = ctypes.c_void_p(256)
    code = lib.spec_verify_stochastic_static(big, _lib.SPEC_BF16, one, one, one, 1.0, one, one, one, one, None, None,
                                             None, None, None, 0.15, None, None, one, None)
    assert code == _lib.SPEC_ERR_TOO_LARGE
    assert b"SPEC_STATIC_SCRATCH_BYTES" in lib.spec_status_str(code)
