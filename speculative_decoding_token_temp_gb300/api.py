"""Torch-facing binding of the C ABI: the same four calls under the same names.

Each function checks dtype, device, contiguity and shapes, allocates the outputs
(unless `out=` passes them in) and the scratch workspace, and calls the C entry
point on the current CUDA stream with the tensors' data pointers. Every step of
the verification itself runs in the CUDA kernels of libspecverify.so.

Logits are torch.bfloat16 or torch.float32 tensors on a CUDA device, shaped
[rows, V] (packed layout, see include/spec_verify.h) or, for dense batches,
[B, gamma+1, V] / [B, gamma, V]."""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import SpecBatch, check


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return _lib.SPEC_BF16
    if t.dtype == torch.float32:
        return _lib.SPEC_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _need(t: torch.Tensor, name: str, dtype=None, numel=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


class Workspace:
    """Device scratch buffer reused across calls (grown on demand)."""

    def __init__(self):
        self.buf = None

    def get(self, nbytes: int, device) -> torch.Tensor:
        nbytes = max(int(nbytes), 256)
        if self.buf is None or self.buf.numel() < nbytes or self.buf.device != device:
            self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        return self.buf


_DEFAULT_WS = {}


def _out(o: dict, name: str, make):
    """o[name], allocated by make() only when the caller has not passed one (no allocation
    on the repeated-call path)."""
    t = o.get(name)
    if t is None:
        t = make()
        o[name] = t
    return t


def _workspace(ws, nbytes, device):
    if isinstance(ws, torch.Tensor):
        if ws.numel() < nbytes:
            raise ValueError(f"workspace has {ws.numel()} bytes, needs {nbytes}")
        return ws
    if ws is None:
        ws = _DEFAULT_WS.setdefault((device.type, device.index), Workspace())
    return ws.get(nbytes, device)


def _geometry(target, draft_rows_or_tokens, cu_draft, gamma, has_bonus=True):
    """(B, gamma_max, V, total_draft, cu pointer, 2-D target view)."""
    V = target.shape[-1]
    if cu_draft is None:
        if target.dim() == 3:
            B = target.shape[0]
            g = target.shape[1] - (1 if has_bonus else 0)
        else:
            if gamma is None:
                raise ValueError("a 2-D dense target needs gamma")
            g = int(gamma)
            rows = target.shape[0]
            B = rows // (g + 1) if has_bonus else rows // max(g, 1)
        total = B * g
        return B, g, V, total, None
    _need(cu_draft, "cu_draft", torch.int32, device=target.device)
    B = cu_draft.numel() - 1
    if gamma is None:
        raise ValueError("packed batches need gamma (an upper bound on every gamma_b)")
    total = int(draft_rows_or_tokens.numel()) if draft_rows_or_tokens is not None else None
    return B, int(gamma), V, total, cu_draft


def spec_workspace_bytes(B: int, gamma: int, V: int, total_draft: int, mode: int, dtype: int = _lib.SPEC_BF16,
                         packed: bool = False) -> int:
    g = SpecBatch(B, gamma, V, total_draft, ctypes.c_void_p(1) if packed else None)
    return int(_lib.lib().spec_workspace_bytes(g, dtype, mode))


def spec_verify_stochastic(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor,
                           temperature: float, u_accept: torch.Tensor, u_sample: torch.Tensor, *,
                           cu_draft: torch.Tensor | None = None, gamma: int | None = None,
                           nkl_delta: float = 0.15, want_probs: bool = True, want_nkl: bool = True,
                           want_greedy: bool = True, out: dict | None = None, workspace=None,
                           device_status: torch.Tensor | None = None, _options: dict | None = None,
                           _static: bool = False) -> dict:
    """Stochastic verification with residual / bonus resampling; see spec_verify.h.

    Returns a dict of device tensors: n_accepted [B], out_tokens [total_draft+B] (dense:
    [B, gamma+1]), and optionally p_x, q_x, alpha, nkl, nkl_mask, greedy_n,
    greedy_tokens, plus device_status [1] (sticky error bits)."""
    dt = _dtype_code(target)
    dev = target.device
    B, g, V, total, cu = _geometry(target, draft_tokens, cu_draft, gamma)
    rows = total + B
    _need(target, "target", target.dtype, rows * V, dev)
    if total > 0:
        _need(draft, "draft", target.dtype, total * V, dev)
    _need(draft_tokens, "draft_tokens", torch.int32, total, dev)
    _need(u_accept, "u_accept", torch.float32, total, dev)
    _need(u_sample, "u_sample", torch.float32, B, dev)
    o = {} if out is None else out

    def get(name, n, dtype):
        t = o.get(name)
        if t is None:
            t = torch.empty(n, dtype=dtype, device=dev)
            o[name] = t
        _need(t, name, dtype, n, dev)
        return t

    n_acc = get("n_accepted", B, torch.int32)
    out_tok = get("out_tokens", rows, torch.int32)
    p_x = get("p_x", total, torch.float32) if want_probs else None
    q_x = get("q_x", total, torch.float32) if want_probs else None
    alpha = get("alpha", total, torch.float32) if want_probs else None
    nkl = get("nkl", total, torch.float32) if want_nkl else None
    mask = get("nkl_mask", total, torch.uint8) if want_nkl else None
    g_n = get("greedy_n", B, torch.int32) if want_greedy else None
    g_tok = get("greedy_tokens", rows, torch.int32) if want_greedy else None
    if device_status is None:
        device_status = o.get("device_status")
        if device_status is None:
            device_status = torch.zeros(1, dtype=torch.int32, device=dev)
    o["device_status"] = device_status
    gb = SpecBatch(B, g, V, total, _ptr(cu))
    args = (gb, dt, _ptr(target), _ptr(draft) if total > 0 else None, _ptr(draft_tokens), float(temperature),
            _ptr(u_accept), _ptr(u_sample), _ptr(n_acc), _ptr(out_tok), _ptr(p_x), _ptr(q_x), _ptr(alpha),
            _ptr(nkl), _ptr(mask), float(nkl_delta), _ptr(g_n), _ptr(g_tok))
    if _static:
        if _options is not None or workspace is not None:
            raise ValueError("the static-scratch call takes neither options nor a workspace")
        code = _lib.lib().spec_verify_stochastic_static(*args, _ptr(device_status), _stream(dev))
        check("spec_verify_stochastic_static", code)
        return o
    nbytes = int(_lib.lib().spec_workspace_bytes(gb, dt, _lib.SPEC_MODE_STOCHASTIC))
    ws = _workspace(workspace, nbytes, dev)
    tail = (_ptr(device_status), _ptr(ws), ws.numel(), _stream(dev))
    if _options is None:
        code = _lib.lib().spec_verify_stochastic(*args, *tail)
        check("spec_verify_stochastic", code)
    else:
        opts = _fill_options(_options, o, dev, B, total)
        code = _lib.lib().spec_verify_stochastic_ex(*args, ctypes.byref(opts), *tail)
        check("spec_verify_stochastic_ex", code)
    return o


def spec_verify_stochastic_static(target, draft, draft_tokens, temperature, u_accept, u_sample, **kw) -> dict:
    """spec_verify_stochastic on the library's static device scratch instead of a workspace
    (for callers that cannot allocate; one such call in flight per GPU); see spec_verify.h."""
    return spec_verify_stochastic(target, draft, draft_tokens, temperature, u_accept, u_sample, _static=True, **kw)


def spec_verify_greedy(target: torch.Tensor, draft_tokens: torch.Tensor, *, cu_draft=None, gamma=None,
                       out: dict | None = None, workspace=None, device_status=None,
                       _options: dict | None = None) -> dict:
    """Greedy argmax-match verification; returns n_accepted [B], out_tokens [total_draft+B]."""
    dt = _dtype_code(target)
    dev = target.device
    B, g, V, total, cu = _geometry(target, draft_tokens, cu_draft, gamma)
    rows = total + B
    _need(target, "target", target.dtype, rows * V, dev)
    _need(draft_tokens, "draft_tokens", torch.int32, total, dev)
    o = {} if out is None else out
    n_acc = _out(o, "n_accepted", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    out_tok = _out(o, "out_tokens", lambda: torch.empty(rows, dtype=torch.int32, device=dev))
    _need(n_acc, "n_accepted", torch.int32, B, dev)
    _need(out_tok, "out_tokens", torch.int32, rows, dev)
    if device_status is None:
        device_status = o.get("device_status")
        if device_status is None:
            device_status = torch.zeros(1, dtype=torch.int32, device=dev)
    o["device_status"] = device_status
    gb = SpecBatch(B, g, V, total, _ptr(cu))
    nbytes = int(_lib.lib().spec_workspace_bytes(gb, dt, _lib.SPEC_MODE_GREEDY))
    ws = _workspace(workspace, nbytes, dev)
    args = (gb, dt, _ptr(target), _ptr(draft_tokens), _ptr(n_acc), _ptr(out_tok))
    tail = (_ptr(device_status), _ptr(ws), ws.numel(), _stream(dev))
    if _options is None:
        check("spec_verify_greedy", _lib.lib().spec_verify_greedy(*args, *tail))
    else:
        opts = _fill_options(_options, o, dev, B, total)
        check("spec_verify_greedy_ex", _lib.lib().spec_verify_greedy_ex(*args, ctypes.byref(opts), *tail))
    return o


def spec_tree_workspace_bytes(B: int, N: int, V: int) -> int:
    """Workspace bytes of spec_verify_tree for B sequences of N nodes over V tokens (0 when
    the geometry is invalid)."""
    return int(_lib.lib().spec_tree_workspace_bytes(int(B), int(N), int(V)))


def spec_status_str(code: int) -> str:
    """The library's description of a spec_status value."""
    return _lib.lib().spec_status_str(int(code)).decode()


def spec_selftest_wait_timeout(device=None, *, device_status: torch.Tensor | None = None) -> torch.Tensor:
    """The failure-detection self-test: the sampler's bounded wait runs against a decision
    that nothing publishes and gives up after its limit. Returns the device status word
    (SPEC_DEV_TIMEOUT set once the stream has reached it); see spec_verify.h."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    if device_status is None:
        device_status = torch.zeros(1, dtype=torch.int32, device=dev)
    _need(device_status, "device_status", torch.int32, 1, dev)
    g = SpecBatch(1, 1, 8, 1, None)
    nbytes = int(_lib.lib().spec_workspace_bytes(g, _lib.SPEC_BF16, _lib.SPEC_MODE_STOCHASTIC))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    code = _lib.lib().spec_selftest_wait_timeout(_ptr(device_status), _ptr(ws), ws.numel(), _stream(dev))
    check("spec_selftest_wait_timeout", code)
    # the workspace stays referenced until the stream has passed the self-test
    torch.cuda.current_stream(dev).synchronize()
    return device_status


def spec_tree_depth(parent) -> int:
    arr = (ctypes.c_int32 * len(parent))(*[int(x) for x in parent])
    return int(_lib.lib().spec_tree_depth(ctypes.cast(arr, ctypes.c_void_p), len(parent)))


def spec_verify_tree(target: torch.Tensor, node_tokens: torch.Tensor, parent, *, out: dict | None = None,
                     workspace=None, device_status=None) -> dict:
    """Greedy tree verification. target [B*(N+1), V] or [B, N+1, V]; node_tokens [B, N] int32;
    parent: host sequence of N ints. Returns accept_len [B], path_nodes [B, D], out_tokens [B, D+1]."""
    dt = _dtype_code(target)
    dev = target.device
    N = len(parent)
    D = spec_tree_depth(parent)
    if D < 1:
        raise ValueError("parent must be a topologically ordered forest of 1..64 nodes")
    B = node_tokens.shape[0] if node_tokens.dim() == 2 else node_tokens.numel() // max(N, 1)
    V = target.shape[-1]
    _need(target, "target", target.dtype, B * (N + 1) * V, dev)
    _need(node_tokens, "node_tokens", torch.int32, B * N, dev)
    o = {} if out is None else out
    acc = _out(o, "accept_len", lambda: torch.empty(B, dtype=torch.int32, device=dev))
    path = _out(o, "path_nodes", lambda: torch.empty(B, D, dtype=torch.int32, device=dev))
    tok = _out(o, "out_tokens", lambda: torch.empty(B, D + 1, dtype=torch.int32, device=dev))
    if device_status is None:
        device_status = o.get("device_status")
        if device_status is None:
            device_status = torch.zeros(1, dtype=torch.int32, device=dev)
    o["device_status"] = device_status
    nbytes = int(_lib.lib().spec_tree_workspace_bytes(B, N, V))
    ws = _workspace(workspace, nbytes, dev)
    par = (ctypes.c_int32 * N)(*[int(x) for x in parent])
    code = _lib.lib().spec_verify_tree(B, N, V, dt, _ptr(target), _ptr(node_tokens),
                                       ctypes.cast(par, ctypes.c_void_p), _ptr(acc), _ptr(path), _ptr(tok),
                                       _ptr(device_status), _ptr(ws), ws.numel(), _stream(dev))
    check("spec_verify_tree", code)
    return o


def spec_nkl(target: torch.Tensor, draft: torch.Tensor, temperature: float, *, cu_draft=None, gamma=None,
             delta: float = 0.15, want_mask: bool = True, out: dict | None = None, workspace=None,
             device_status=None, _options: dict | None = None) -> dict:
    """NKL = KL(q||p)/ln V per (target row i, draft row i); returns nkl [total_draft], nkl_mask."""
    dt = _dtype_code(target)
    dev = target.device
    B, g, V, total, cu = _geometry(target, draft, cu_draft, gamma)
    if cu is not None:
        total = draft.numel() // V
    _need(target, "target", target.dtype, (total + B) * V, dev)
    _need(draft, "draft", target.dtype, total * V, dev)
    o = {} if out is None else out
    nkl = _out(o, "nkl", lambda: torch.empty(total, dtype=torch.float32, device=dev))
    mask = _out(o, "nkl_mask", lambda: torch.empty(total, dtype=torch.uint8, device=dev)) if want_mask else None
    if device_status is None:
        device_status = o.get("device_status")
        if device_status is None:
            device_status = torch.zeros(1, dtype=torch.int32, device=dev)
    o["device_status"] = device_status
    gb = SpecBatch(B, g, V, total, _ptr(cu))
    nbytes = int(_lib.lib().spec_workspace_bytes(gb, dt, _lib.SPEC_MODE_NKL))
    ws = _workspace(workspace, nbytes, dev)
    args = (gb, dt, _ptr(target), _ptr(draft), float(temperature), float(delta), _ptr(nkl), _ptr(mask))
    tail = (_ptr(device_status), _ptr(ws), ws.numel(), _stream(dev))
    if _options is None:
        check("spec_nkl", _lib.lib().spec_nkl(*args, *tail))
    else:
        opts = _fill_options(_options, o, dev, B, total)
        check("spec_nkl_ex", _lib.lib().spec_nkl_ex(*args, ctypes.byref(opts), *tail))
    return o


# ---------------------------------------------------------------------------
# policy variants (spec_options)

def _fill_options(opt: dict, o: dict, dev, B: int, total: int) -> _lib.SpecOptions:
    """A spec_options block from keyword options; block-accept outputs are allocated into o."""
    so = _lib.SpecOptions()
    so.temperature_draft = float(opt.get("temperature_draft", 0.0))
    pos = opt.get("position")
    if pos is not None:
        _need(pos, "position", torch.int32, B, dev)
        so.position = pos.data_ptr()
    so.delta_alpha = float(opt.get("delta_alpha", 0.08))
    so.delta_max = float(opt.get("delta_max", 0.3))
    mb = int(opt.get("min_block_len", 0))
    so.min_block_len = mb
    if mb > 0:
        bn = _out(o, "block_n", lambda: torch.empty(B, dtype=torch.int32, device=dev))
        bt = _out(o, "block_tokens", lambda: torch.empty(total, dtype=torch.int32, device=dev))
        _need(bn, "block_n", torch.int32, B, dev)
        _need(bt, "block_tokens", torch.int32, total, dev)
        so.block_n = bn.data_ptr()
        so.block_tokens = bt.data_ptr() if total > 0 else None
    st = opt.get("stats")
    if st is not None:
        _need(st, "stats", torch.uint8, _lib.STATS_BYTES, dev)
        so.stats = st.data_ptr()
        so.stats_bucket = int(opt.get("stats_bucket", 0))
    return so


_OPTION_KEYS = ("temperature_draft", "position", "delta_alpha", "delta_max", "min_block_len", "stats",
                "stats_bucket")


def _split(kw: dict):
    opts = {k: kw.pop(k) for k in list(kw) if k in _OPTION_KEYS}
    return opts, kw


def spec_verify_stochastic_ex(target, draft, draft_tokens, temperature, u_accept, u_sample, **kw) -> dict:
    """spec_verify_stochastic with spec_options: temperature_draft (T_d, 0 = T), position [B]
    int32 (1-based position of each sequence's first draft; position-adaptive NKL mask),
    delta_alpha, delta_max, min_block_len (block-accept: block_n [B], block_tokens
    [total_draft] in the result), stats (a new_accept_stats() buffer) and stats_bucket."""
    opts, kw = _split(dict(kw))
    return spec_verify_stochastic(target, draft, draft_tokens, temperature, u_accept, u_sample, _options=opts, **kw)


def spec_verify_greedy_ex(target, draft_tokens, **kw) -> dict:
    """spec_verify_greedy with spec_options (min_block_len, stats, stats_bucket)."""
    opts, kw = _split(dict(kw))
    return spec_verify_greedy(target, draft_tokens, _options=opts, **kw)


def spec_nkl_ex(target, draft, temperature, **kw) -> dict:
    """spec_nkl with spec_options (position, delta_alpha, delta_max)."""
    opts, kw = _split(dict(kw))
    return spec_nkl(target, draft, temperature, _options=opts, **kw)


def new_accept_stats(device) -> torch.Tensor:
    """A zero-filled spec_accept_stats buffer on `device` (uint8 [sizeof(spec_accept_stats)])."""
    return torch.zeros(_lib.STATS_BYTES, dtype=torch.uint8, device=device)


def spec_accept_summary(stats: torch.Tensor, bucket_now: int, window: int, out: torch.Tensor | None = None):
    """Device fp64 [6]: rounds, accepted drafts, drafts, mean accepted per round, mean
    acceptance rate, ARSD over the buckets (bucket_now - window, bucket_now]."""
    dev = stats.device
    _need(stats, "stats", torch.uint8, _lib.STATS_BYTES, dev)
    if out is None:
        out = torch.empty(6, dtype=torch.float64, device=dev)
    _need(out, "out", torch.float64, 6, dev)
    check("spec_accept_summary", _lib.lib().spec_accept_summary(_ptr(stats), int(bucket_now), int(window),
                                                                _ptr(out), _stream(dev)))
    return out


# ---------------------------------------------------------------------------
# multi-draft verification

def spec_multi_workspace_bytes(G: int, K: int, gamma: int, V: int, dtype: int = _lib.SPEC_BF16,
                               stochastic: bool = True) -> int:
    return int(_lib.lib().spec_multi_workspace_bytes(_lib.SpecMultiBatch(G, K, gamma, V), dtype, int(stochastic)))


def spec_verify_multi(target: torch.Tensor, draft: torch.Tensor, draft_tokens: torch.Tensor, K: int,
                      temperature: float, *, stochastic: bool = True, u_accept: torch.Tensor | None = None,
                      u_sample: torch.Tensor | None = None, consensus_nkl: float = 0.1, divergence_nkl: float = 0.15,
                      want_matrix: bool = True, out: dict | None = None, workspace=None,
                      device_status=None) -> dict:
    """G groups of K candidates (candidate k of group g is sequence g*K + k of a dense batch):
    target [G*K*(gamma+1), V], draft [G*K*gamma, V], draft_tokens [G*K*gamma] int32. Returns
    n_accepted [G*K], out_tokens [G*K*(gamma+1)], best_k / best_n [G], best_tokens
    [G*(gamma+1)] and, with want_matrix, pair_nkl [G*gamma*K*K], consensus / divergence
    [G*gamma]."""
    dt = _dtype_code(target)
    dev = target.device
    V = target.shape[-1]
    seqs = draft_tokens.numel()
    rows = target.numel() // V
    if K < 2 or (rows - seqs) % K:
        raise ValueError("target rows must be G*K*(gamma+1)")
    G = (rows - seqs) // K
    gamma = seqs // (G * K) if G else 0
    _need(target, "target", target.dtype, G * K * (gamma + 1) * V, dev)
    if gamma:
        _need(draft, "draft", target.dtype, G * K * gamma * V, dev)
    _need(draft_tokens, "draft_tokens", torch.int32, G * K * gamma, dev)
    if stochastic:
        _need(u_sample, "u_sample", torch.float32, G * K, dev)
        _need(u_accept, "u_accept", torch.float32, G * K * gamma, dev)
    o = {} if out is None else out
    i32 = lambda n: torch.empty(n, dtype=torch.int32, device=dev)  # noqa: E731
    n_acc = _out(o, "n_accepted", lambda: i32(G * K))
    out_tok = _out(o, "out_tokens", lambda: i32(G * K * (gamma + 1)))
    bk, bn = _out(o, "best_k", lambda: i32(G)), _out(o, "best_n", lambda: i32(G))
    bt = _out(o, "best_tokens", lambda: i32(G * (gamma + 1)))
    pn = cons = div = None
    if want_matrix:
        pn = _out(o, "pair_nkl", lambda: torch.empty(G * gamma * K * K, dtype=torch.float32, device=dev))
        cons = _out(o, "consensus", lambda: torch.empty(G * gamma, dtype=torch.uint8, device=dev))
        div = _out(o, "divergence", lambda: torch.empty(G * gamma, dtype=torch.uint8, device=dev))
    if device_status is None:
        device_status = o.get("device_status")
        if device_status is None:
            device_status = torch.zeros(1, dtype=torch.int32, device=dev)
    o["device_status"] = device_status
    mb = _lib.SpecMultiBatch(G, K, gamma, V)
    nbytes = int(_lib.lib().spec_multi_workspace_bytes(mb, dt, int(stochastic)))
    ws = _workspace(workspace, nbytes, dev)
    code = _lib.lib().spec_verify_multi(
        mb, dt, int(stochastic), _ptr(target), _ptr(draft) if gamma else None, _ptr(draft_tokens),
        float(temperature), _ptr(u_accept) if stochastic else None, _ptr(u_sample) if stochastic else None,
        float(consensus_nkl), float(divergence_nkl), _ptr(n_acc), _ptr(out_tok), _ptr(bk), _ptr(bn), _ptr(bt),
        _ptr(pn), _ptr(cons), _ptr(div), _ptr(device_status), _ptr(ws), ws.numel(), _stream(dev))
    check("spec_verify_multi", code)
    return o
