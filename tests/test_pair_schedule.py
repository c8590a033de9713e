"""Host-side pins of the many-token projection GEMM's work schedule (no GPU needed): the
library's own planner and item walk (attn_debug_pair_schedule) must cover every output
column of every 256 x 256 tile exactly once, in pieces the kernel can run, and cut a partial
last round so that no pair carries more than its share of it."""
import math

import pytest

from transformer_gqa_attention_gb300 import _build, abi

TOKENS = [1, 65, 128, 200, 256, 300, 512, 1000, 2048, 2100, 4096, 8192, 19456, 32768, 262144]
N_TILES = [24, 16]  # Q/K/V (6144 columns), W_O (4096 columns)
PAIRS = [76, 75, 74, 70, 64, 8, 1]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    _build.build()
    abi.lib()


def _walk(m_tiles, n_tiles, n_pairs):
    full, tail_w, grid, items = abi.attn_debug_pair_schedule(m_tiles, n_tiles, n_pairs)
    return full, tail_w, grid, items


@pytest.mark.parametrize("n_tiles", N_TILES)
@pytest.mark.parametrize("n_pairs", PAIRS)
def test_every_column_covered_once_in_runnable_pieces(n_tiles, n_pairs):
    for n_tok in TOKENS:
        m_tiles = (n_tok + 255) // 256
        full, tail_w, grid, items = _walk(m_tiles, n_tiles, n_pairs)
        assert grid % 2 == 0 and 2 <= grid <= 2 * n_pairs
        seen = {}
        for pair, mt, n0, w in items:
            assert 0 <= pair < grid // 2
            assert 0 <= mt < m_tiles
            # UMMA N = w for M = 256 (a multiple of 16 up to 256), each CTA stages w/2 weight
            # rows, the epilogue works in 32-column chunks that never cross a head slice
            assert w % 32 == 0 and 32 <= w <= 256
            assert n0 % 32 == 0 and 0 <= n0 and n0 + w <= n_tiles * 256
            if w == 256:
                assert n0 % 256 == 0
            for c in range(n0, n0 + w, 32):
                key = (mt, c)
                assert key not in seen, (n_tok, key)
                seen[key] = pair
        assert len(seen) == m_tiles * n_tiles * 8, n_tok


@pytest.mark.parametrize("n_tiles", N_TILES)
def test_partial_last_round_is_spread(n_tiles):
    n_pairs = 76
    for n_tok in TOKENS:
        m_tiles = (n_tok + 255) // 256
        total = m_tiles * n_tiles
        full, tail_w, grid, items = _walk(m_tiles, n_tiles, n_pairs)
        assert full == total // n_pairs
        per_pair = {}
        for pair, mt, n0, w in items:
            per_pair.setdefault(pair, []).append(w)
        if total % n_pairs == 0:
            assert tail_w == 0
        if tail_w:
            assert tail_w % 32 == 0 and tail_w < 256
            # whole tiles first, then at most one piece per pair, none wider than tail_w
            for ws in per_pair.values():
                assert all(w == 256 for w in ws[:full])
                assert len(ws) <= full + 1
                assert all(w <= tail_w for w in ws[full:])
            # the smallest width that fits: each m row of the partial round is cut separately;
            # at tail_w the pieces fit the pairs, one step narrower they would not
            base = full * n_pairs

            def pieces(w):
                r, c, k = base // n_tiles, (base % n_tiles) * 256, 0
                while r < m_tiles:
                    k += math.ceil((n_tiles * 256 - c) / w)
                    r, c = r + 1, 0
                return k
            assert pieces(tail_w) <= n_pairs
            assert tail_w == 32 or pieces(tail_w - 32) > n_pairs
            assert len(items) - full * n_pairs == pieces(tail_w)
            # makespan in tile units: full rounds plus tail_w / 256 instead of one more round
            makespan = max(sum(ws) for ws in per_pair.values()) / 256
            assert makespan <= full + tail_w / 256 + 1e-9
            assert makespan < math.ceil(total / n_pairs)
        else:
            makespan = max(sum(ws) for ws in per_pair.values()) / 256
            assert makespan == math.ceil(total / min(n_pairs, total))


def test_two_thousand_tokens_schedule():
    # 2048 tokens on 76 pairs: Q/K/V 2 whole rounds + 160-column pieces, W_O 1 round + 192
    q = _walk(8, 24, 76)
    o = _walk(8, 16, 76)
    assert q[:3] == (2, 160, 152)
    assert o[:3] == (1, 192, 152)


def test_invalid_arguments_rejected():
    import ctypes
    L = abi.lib()
    i32 = ctypes.c_int
    a, b, c, n = i32(), i32(), i32(), i32()
    assert L.attn_debug_pair_schedule(0, 24, 76, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None, 0,
                                      ctypes.byref(n)) == 1
    assert L.attn_debug_pair_schedule(8, 24, 0, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None, 0,
                                      ctypes.byref(n)) == 1
    assert L.attn_debug_pair_schedule(8, 24, 76, None, ctypes.byref(b), ctypes.byref(c), None, 0,
                                      ctypes.byref(n)) == 1
    # too small an item buffer: GQA_ERR_SHAPE with the count reported
    assert L.attn_debug_pair_schedule(8, 24, 76, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c), None, 0,
                                      ctypes.byref(n)) == 2
    assert n.value > 0
