"""The product path has no CPU fallback: without the built library the binding raises, and
host tensors are refused before anything is launched. No GPU needed."""
import numpy as np
import pytest
import torch

from speculative_decoding_token_temp_gb300 import _lib, api, synth


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_LIB", None)
    monkeypatch.setattr(_lib, "LIB", str(tmp_path / "libspecverify.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _lib.lib()


def test_host_tensors_are_refused():
    w = synth.make_stochastic(2, 64, synth.F32, 1.0, seed=3, gamma=2)
    t = torch.from_numpy(np.ascontiguousarray(w.target))
    d = torch.from_numpy(np.ascontiguousarray(w.draft))
    tok = torch.from_numpy(w.tokens)
    ua, us = torch.from_numpy(w.u_accept), torch.from_numpy(w.u_sample)
    with pytest.raises(ValueError, match="CUDA"):
        api.spec_verify_stochastic(t, d, tok, 1.0, ua, us, gamma=2)
    with pytest.raises(ValueError, match="CUDA"):
        api.spec_verify_greedy(t, tok, gamma=2)
    with pytest.raises(ValueError, match="CUDA"):
        api.spec_nkl(t, d, 1.0, gamma=2)
