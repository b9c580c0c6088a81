"""Host-side launch planning (csrc/plan.h) at several SM counts, without a GPU: the
header is compiled with g++ through tests/plan_driver.cpp and queried for the vocabulary
chunking of the tile kernels and the sampler's ranges. The chunking must cover every
token once in chunks that start on 16-byte boundaries, split only while the grid still
fits in one wave, never below 8192 tokens, and grow monotonically with the wave; the
sampler's ranges must cover every stage once inside one wave. On a GB300 (152 SMs, four
resident tile blocks each) the plans are the ones the kernels were tuned with."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "speculative_decoding_token_temp_gb300", "csrc")


@pytest.fixture(scope="module")
def plan(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ not found")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_driver")
    subprocess.run([gxx, "-std=c++17", "-O1", "-I", CSRC, os.path.join(HERE, "plan_driver.cpp"), "-o", exe],
                   check=True, capture_output=True)

    def query(lines):
        out = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True, check=True)
        return [tuple(int(x) for x in l.split()) for l in out.stdout.strip().splitlines()]
    return query


SLOTS = sorted([1, 76 * 2, 132 * 4, 148 * 4, 152 * 2, 152 * 4, 160 * 4, 264 * 4, 4096, 10000])
CASES = [  # V, rows (tiles per chunk), max_chunk
    (128256, 2304, 65536), (128256, 2048, 49152), (32000, 384, 65536), (128256, 416, 65536),
    (152064, 4985, 65536), (128256, 48, 65536), (1000, 1, 65536), (1 << 20, 3, 65536), (50257, 320, 65536),
    (128256, 64 * 9, 131072), (8, 1, 65536), (8192 * 3 + 5, 2, 65536),
]


def test_chunking_covers_the_row_within_one_wave(plan):
    q = [f"chunk {V} {rows} {mc} {s}" for V, rows, mc in CASES for s in SLOTS]
    res = iter(plan(q))
    for V, rows, mc in CASES:
        prev = 0
        for s in SLOTS:
            n, ce = next(res)
            assert ce % 8 == 0 and ce > 0, (V, rows, s)
            assert (n - 1) * ce < V <= n * ce, (V, rows, s, n, ce)       # every token in exactly one chunk
            base = -(-V // mc)
            if n > base:                                                  # split beyond max_chunk only ...
                assert rows * n <= min(s, 4096), (V, rows, s, n)          # ... while the grid fits one wave
                assert V // n >= 8192 - 8, (V, rows, s, n)                # ... and not below 8192 tokens
            assert n >= prev, (V, rows, s)                                # more slots never mean fewer chunks
            prev = n


def test_chunking_on_a_gb300_matches_the_tuned_plans(plan):
    # 152 SMs x 4 resident tile blocks: the headline's pair tiles are 2 chunks of 64128
    # tokens (4608 tiles), the tree's rows 2 chunks (832 tiles), the B=64 / V=32000 rows whole
    gb300 = 152 * 4
    got = plan([f"chunk 128256 2304 65536 {gb300}", f"chunk 128256 416 65536 {gb300}",
                f"chunk 32000 384 65536 {gb300}", f"chunk 128256 48 65536 {gb300}"])
    assert got[0] == (2, 64128)
    assert got[1] == (2, 64128)
    assert got[2] == (1, 32000)
    assert got[3][0] == 12                       # B=8, gamma=5: split to 576 tiles, under one wave


@pytest.mark.parametrize("wave", [1, 3, 4, 152 * 4, 132 * 4, 264 * 4])
def test_sampler_ranges_cover_every_stage_once_in_one_wave(plan, wave):
    shapes = [(256, 32), (64, 8), (512, 38), (1, 1), (3, 200), (16, 32), (17, 5), (0, 4)]
    res = plan([f"sampler {B} {nst} {wave} 16 1" for B, nst in shapes])
    for (B, nst), (head_total, nb_head, seg_head, nb_tail, seg_tail) in zip(shapes, res):
        total = B * nst
        assert head_total == max(B - 16, 0) * nst
        covered = []
        for k in range(nb_head):
            covered += list(range(k * seg_head, min(head_total, (k + 1) * seg_head)))
        for k in range(nb_tail):
            lo = head_total + k * seg_tail
            covered += list(range(lo, min(total, lo + seg_tail)))
        assert covered == list(range(total)), (B, nst, wave)
        assert all(k * seg_head < head_total for k in range(nb_head))       # no empty block
        if wave >= 2:
            assert nb_head + nb_tail <= wave, (B, nst, wave, nb_head, nb_tail)
        assert nb_tail <= max(wave // 4, 1)
