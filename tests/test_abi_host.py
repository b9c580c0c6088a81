"""The C-ABI library loads and exports what include/spec_verify.h declares; host-side
argument checks and workspace sizing. No GPU: nothing here launches a kernel."""
import ctypes

import pytest

from speculative_decoding_token_temp_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.lib()


def test_every_declared_symbol_is_exported(lib):
    names = _lib.declared_functions()
    assert {"spec_verify_stochastic", "spec_verify_greedy", "spec_verify_tree", "spec_nkl",
            "spec_workspace_bytes", "spec_tree_workspace_bytes", "spec_tree_depth", "spec_status_str"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
    assert set(_lib.SIGNATURES) >= set(names)


def test_bounds_checked_variant_exports_the_same_symbols(lib):
    """The debug build (every computed access checked against its buffer) has the same ABI."""
    checked = _lib.bounds_lib()
    for n in _lib.declared_functions():
        assert hasattr(checked, n), n
    assert _lib.SPEC_DEV_BOUNDS not in (_lib.SPEC_DEV_TOKEN_RANGE, _lib.SPEC_DEV_NONFINITE, _lib.SPEC_DEV_OFFSETS,
                                        _lib.SPEC_DEV_TIMEOUT, _lib.SPEC_DEV_POSITION)


def test_status_strings(lib):
    assert lib.spec_status_str(0) == b"ok"
    assert b"workspace" in lib.spec_status_str(3)


def _g(B, gamma, V, total=None, cu=None):
    return _lib.SpecBatch(B, gamma, V, B * gamma if total is None else total, cu)


def test_workspace_sizes(lib):
    BF, F = _lib.SPEC_BF16, _lib.SPEC_F32
    h = lib.spec_workspace_bytes(_g(256, 8, 128256), BF, _lib.SPEC_MODE_STOCHASTIC)
    # 2304 rows x 2 chunks (of at most 65536 tokens) x 32 B partials, tickets, records,
    # and the sampler's slice-mass table: 256 sequences x 32 stages x 16 slices x 4 B
    table = 256 * 32 * 16 * 4
    assert 2304 * 2 * 32 + table <= h < 2304 * 2 * 32 + table + 256 * 200
    assert lib.spec_workspace_bytes(_g(256, 8, 128256), F, _lib.SPEC_MODE_STOCHASTIC) > h   # f32: twice the table
    assert lib.spec_workspace_bytes(_g(256, 8, 128256), BF, _lib.SPEC_MODE_GREEDY) <= h
    assert lib.spec_workspace_bytes(_g(0, 8, 100), BF, _lib.SPEC_MODE_STOCHASTIC) >= 0
    assert lib.spec_workspace_bytes(_g(2, 200, 100), BF, 0) == 0        # gamma above the limit
    assert lib.spec_workspace_bytes(_g(2, 8, 100), 9, 0) == 0           # unknown dtype
    assert lib.spec_tree_workspace_bytes(32, 12, 128256) > 0
    assert lib.spec_tree_workspace_bytes(32, 65, 128256) == 0


def _tree_depth(lib, parent):
    arr = (ctypes.c_int32 * len(parent))(*parent)
    return lib.spec_tree_depth(ctypes.cast(arr, ctypes.c_void_p), len(parent))


def test_tree_depth(lib):
    assert _tree_depth(lib, [-1, -1, -1, 0, 1, 2, 3, 4, 5, 6, 7, 8]) == 4
    assert _tree_depth(lib, [-1, 0, 1, 2]) == 4
    assert _tree_depth(lib, [-1, 1]) == -1        # not topologically ordered
    assert _tree_depth(lib, [0]) == -1


def test_host_validation_without_launch(lib):
    """Every rejected argument returns before any CUDA call, so this runs without a GPU."""
    P = ctypes.c_void_p
    one = P(256)
    args = dict(dt=_lib.SPEC_BF16, T=0.6)

    def stoch(g, dt=_lib.SPEC_BF16, T=0.6, ws=one, wsb=1 << 30, target=one, status=one):
        return lib.spec_verify_stochastic(g, dt, target, one, one, T, one, one, one, one, None, None, None, None,
                                          None, 0.15, None, None, status, ws, wsb, None)

    g = _g(4, 3, 1000)
    assert stoch(g, dt=7) == _lib.SPEC_ERR_DTYPE
    assert stoch(g, T=0.0) == _lib.SPEC_ERR_INVALID_ARG
    assert stoch(g, T=float("nan")) == _lib.SPEC_ERR_INVALID_ARG
    assert stoch(g, T=-1.0) == _lib.SPEC_ERR_INVALID_ARG
    assert stoch(g, target=None) == _lib.SPEC_ERR_INVALID_ARG
    assert stoch(g, status=None) == _lib.SPEC_ERR_INVALID_ARG
    assert stoch(g, ws=None) == _lib.SPEC_ERR_WORKSPACE
    assert stoch(g, wsb=16) == _lib.SPEC_ERR_WORKSPACE
    assert stoch(g, ws=P(257)) == _lib.SPEC_ERR_WORKSPACE           # not 256-byte aligned
    assert stoch(_g(4, 3, 1000, total=11)) == _lib.SPEC_ERR_INVALID_ARG   # dense total != B*gamma
    assert stoch(_g(4, 3, 0)) == _lib.SPEC_ERR_INVALID_ARG
    assert stoch(_g(4, 129, 10)) == _lib.SPEC_ERR_INVALID_ARG
    assert stoch(_g(0, 3, 10)) == _lib.SPEC_OK                       # empty batch: nothing to do
    assert lib.spec_verify_greedy(g, 5, one, one, one, one, one, one, 1 << 30, None) == _lib.SPEC_ERR_DTYPE
    assert lib.spec_nkl(g, _lib.SPEC_F32, one, one, 0.0, 0.15, one, None, one, one, 1 << 30, None) == \
        _lib.SPEC_ERR_INVALID_ARG
    # every pointer on its element's grid
    assert stoch(g, target=P(257)) == _lib.SPEC_ERR_INVALID_ARG                    # bf16 logits: 2 bytes
    assert stoch(g, dt=_lib.SPEC_F32, target=P(258)) == _lib.SPEC_ERR_INVALID_ARG  # fp32 logits: 4 bytes
    assert stoch(g, status=P(258)) == _lib.SPEC_ERR_INVALID_ARG                    # 32-bit words: 4 bytes
    assert lib.spec_verify_greedy(g, _lib.SPEC_BF16, P(257), one, one, one, one, one, 1 << 30, None) == \
        _lib.SPEC_ERR_INVALID_ARG
    assert lib.spec_verify_greedy(g, _lib.SPEC_BF16, one, P(258), one, one, one, one, 1 << 30, None) == \
        _lib.SPEC_ERR_INVALID_ARG
    assert lib.spec_nkl(g, _lib.SPEC_F32, one, P(258), 0.7, 0.15, one, None, one, one, 1 << 30, None) == \
        _lib.SPEC_ERR_INVALID_ARG
    chain = (ctypes.c_int32 * 2)(-1, 0)
    assert lib.spec_verify_tree(2, 2, 100, _lib.SPEC_BF16, P(257), one, ctypes.cast(chain, P), one, one, one,
                                one, one, 1 << 30, None) == _lib.SPEC_ERR_INVALID_ARG
    out = (ctypes.c_double * 6)()
    assert lib.spec_accept_summary(P(260), 0, 4, ctypes.cast(out, P), None) == _lib.SPEC_ERR_INVALID_ARG
    assert lib.spec_selftest_wait_timeout(None, one, 1 << 30, None) == _lib.SPEC_ERR_INVALID_ARG
    assert lib.spec_selftest_wait_timeout(P(258), one, 1 << 30, None) == _lib.SPEC_ERR_INVALID_ARG
    assert lib.spec_selftest_wait_timeout(one, None, 1 << 30, None) == _lib.SPEC_ERR_WORKSPACE
    assert lib.spec_selftest_wait_timeout(one, one, 16, None) == _lib.SPEC_ERR_WORKSPACE
    bad_parent = (ctypes.c_int32 * 2)(-1, 5)
    assert lib.spec_verify_tree(2, 2, 100, _lib.SPEC_BF16, one, one, ctypes.cast(bad_parent, P), one, one, one,
                                one, one, 1 << 30, None) == _lib.SPEC_ERR_INVALID_ARG


def test_option_checks_without_launch(lib):
    """Options are checked before anything is launched: a bad draft temperature, block-accept
    without its outputs, a non-finite threshold parameter, a bad summary window."""
    P = ctypes.c_void_p
    one = P(256)
    g = _g(4, 3, 1000)

    def stoch(opts, T=0.6):
        return lib.spec_verify_stochastic_ex(g, _lib.SPEC_BF16, one, one, one, T, one, one, one, one, None, None,
                                             None, None, None, 0.15, None, None, ctypes.byref(opts), one, None,
                                             1 << 30, None)

    def greedy(opts):
        return lib.spec_verify_greedy_ex(g, _lib.SPEC_BF16, one, one, one, one, ctypes.byref(opts), one, None,
                                         1 << 30, None)

    o = _lib.SpecOptions()
    o.temperature_draft = -0.5
    assert stoch(o) == _lib.SPEC_ERR_INVALID_ARG
    o.temperature_draft = float("inf")
    assert stoch(o) == _lib.SPEC_ERR_INVALID_ARG
    o = _lib.SpecOptions()
    o.min_block_len = 3
    assert stoch(o) == _lib.SPEC_ERR_INVALID_ARG           # block_n / block_tokens missing
    assert greedy(o) == _lib.SPEC_ERR_INVALID_ARG
    o.min_block_len = -1
    assert greedy(o) == _lib.SPEC_ERR_INVALID_ARG
    o = _lib.SpecOptions()
    o.position = 256
    o.delta_alpha = float("nan")
    assert stoch(o) == _lib.SPEC_ERR_INVALID_ARG
    assert lib.spec_nkl_ex(g, _lib.SPEC_BF16, one, one, 0.6, 0.15, one, None, ctypes.byref(o), one, None, 1 << 30,
                           None) == _lib.SPEC_ERR_INVALID_ARG
    assert greedy(o) == _lib.SPEC_ERR_WORKSPACE            # greedy ignores the position fields
    assert lib.spec_accept_summary(one, 5, 0, one, None) == _lib.SPEC_ERR_INVALID_ARG
    assert lib.spec_accept_summary(one, 5, _lib.SPEC_STATS_SLOTS + 1, one, None) == _lib.SPEC_ERR_INVALID_ARG
    assert lib.spec_accept_summary(None, 5, 4, one, None) == _lib.SPEC_ERR_INVALID_ARG
    o = _lib.SpecOptions()
    o.position = 258                                       # int32 array off its 4-byte grid
    assert stoch(o) == _lib.SPEC_ERR_INVALID_ARG
    o = _lib.SpecOptions()
    o.stats = 260                                          # 64-bit counters off their 8-byte grid
    assert greedy(o) == _lib.SPEC_ERR_INVALID_ARG
    # block-accept outputs of no elements may be NULL: block_tokens when no sequence has a
    # draft (the options pass; the missing workspace is the next check), both when B = 0
    o = _lib.SpecOptions()
    o.min_block_len = 3
    o.block_n = 256
    g0 = _g(4, 0, 1000)
    assert lib.spec_verify_stochastic_ex(g0, _lib.SPEC_BF16, one, None, None, 0.6, None, one, one, one, None, None,
                                         None, None, None, 0.15, None, None, ctypes.byref(o), one, None, 1 << 30,
                                         None) == _lib.SPEC_ERR_WORKSPACE
    assert lib.spec_verify_greedy_ex(g0, _lib.SPEC_BF16, one, None, one, one, ctypes.byref(o), one, None, 1 << 30,
                                     None) == _lib.SPEC_ERR_WORKSPACE
    o.block_n = None
    assert lib.spec_verify_greedy_ex(g0, _lib.SPEC_BF16, one, None, one, one, ctypes.byref(o), one, None, 1 << 30,
                                     None) == _lib.SPEC_ERR_INVALID_ARG   # B = 4 sequences: block_n needed
    assert lib.spec_verify_greedy_ex(_g(0, 3, 1000), _lib.SPEC_BF16, one, None, one, one, ctypes.byref(o), one,
                                     None, 1 << 30, None) == _lib.SPEC_OK


def test_option_structs_match_the_header(tmp_path):
    """The ctypes mirrors of spec_options and spec_accept_stats have the C layout (sizes and
    offsets printed by a program compiled against the header)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    src = tmp_path / "layout.c"
    src.write_text('''#include <stdio.h>
#include <stddef.h>
#include "spec_verify.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\\n", sizeof(spec_options), sizeof(spec_accept_stats),
         offsetof(spec_options, position), offsetof(spec_options, delta_alpha), offsetof(spec_options, min_block_len),
         offsetof(spec_options, block_n), offsetof(spec_options, block_tokens), offsetof(spec_options, stats),
         offsetof(spec_options, stats_bucket), sizeof(spec_stats_slot), offsetof(spec_stats_slot, rate2_fx));
  return 0;
}
''')
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", build.INCLUDE, "-o", str(exe), str(src)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    O, S = _lib.SpecOptions, _lib.SpecStatsSlot
    want = [ctypes.sizeof(O), _lib.STATS_BYTES, O.position.offset, O.delta_alpha.offset, O.min_block_len.offset,
            O.block_n.offset, O.block_tokens.offset, O.stats.offset, O.stats_bucket.offset, ctypes.sizeof(S),
            S.rate2_fx.offset]
    assert got == want


def test_multi_draft_checks_without_launch(lib):
    P = ctypes.c_void_p
    one = P(256)

    def multi(G=4, K=3, gamma=2, V=1000, stochastic=1, T=0.8, ws=one, wsb=1 << 30, c=0.1, d=0.15, ua=one):
        m = _lib.SpecMultiBatch(G, K, gamma, V)
        return lib.spec_verify_multi(m, _lib.SPEC_BF16, stochastic, one, one, one, T, ua, one, c, d, one, one, one,
                                     one, one, None, None, None, one, ws, wsb, None)

    assert multi(K=1) == _lib.SPEC_ERR_INVALID_ARG
    assert multi(K=_lib.SPEC_MAX_CANDIDATES + 1) == _lib.SPEC_ERR_INVALID_ARG
    assert multi(gamma=_lib.SPEC_MAX_GAMMA + 1) == _lib.SPEC_ERR_INVALID_ARG
    assert multi(T=0.0) == _lib.SPEC_ERR_INVALID_ARG
    assert multi(c=float("nan")) == _lib.SPEC_ERR_INVALID_ARG
    assert multi(ua=None) == _lib.SPEC_ERR_INVALID_ARG          # stochastic needs u_accept
    assert multi(ws=None) == _lib.SPEC_ERR_WORKSPACE
    assert multi(wsb=1024) == _lib.SPEC_ERR_WORKSPACE
    assert multi(G=0) == _lib.SPEC_OK
    mb = _lib.SpecMultiBatch(64, 3, 8, 128256)
    sto = lib.spec_multi_workspace_bytes(mb, _lib.SPEC_BF16, 1)
    single = lib.spec_workspace_bytes(_g(192, 8, 128256), _lib.SPEC_BF16, _lib.SPEC_MODE_STOCHASTIC)
    assert sto > single and lib.spec_multi_workspace_bytes(mb, _lib.SPEC_BF16, 0) < sto
    assert lib.spec_multi_workspace_bytes(_lib.SpecMultiBatch(4, 1, 2, 100), _lib.SPEC_BF16, 1) == 0


def test_python_binding_names_every_entry_point(lib):
    """The binding has a same-named function for every entry point the header declares;
    the host-only ones answer without a GPU."""
    from speculative_decoding_token_temp_gb300 import api
    assert [n for n in _lib.declared_functions() if not callable(getattr(api, n, None))] == []
    assert api.spec_status_str(0) == "ok"
    assert "workspace" in api.spec_status_str(_lib.SPEC_ERR_WORKSPACE)
    assert api.spec_tree_workspace_bytes(32, 12, 128256) == lib.spec_tree_workspace_bytes(32, 12, 128256) > 0
    assert api.spec_tree_workspace_bytes(32, 65, 128256) == 0
    assert api.spec_tree_depth([-1, -1, -1, 0, 1, 2, 3, 4, 5, 6, 7, 8]) == 4
