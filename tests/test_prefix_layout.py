"""Host-side index construction of the shared-prefix decode (no GPU)."""
import numpy as np
import pytest

import workloads as W
from sm_load_balancing_gb300.prefix import shared_prefix_layout


def _w(seqlens, groups, lens, T=1, Hq=8, Hkv=2, P=16):
    w = W.make_custom(seqlens, q_tokens=T, num_q_heads=Hq, num_kv_heads=Hkv, head_dim_qk=16, page_size=P, seed=1)
    return W.share_prefix(w, groups, lens)


def test_rows_map_each_request_row_to_its_stacked_prefix_row():
    w = _w([100, 70, 90, 40, 120, 66], [[0, 2, 3, 4, 5], [1]], [32, 48])
    lay = shared_prefix_layout(w.seqlens, w.page_table, w.prefix_groups, w.prefix_lens, 16, 1, 8, 2)
    R = lay.rows_per_virtual
    assert R == 16 // 4  # G = 4, T = 1
    # group 0 has 5 members -> two virtual requests, group 1 one
    assert [v for v in lay.virtual] == [(0, [0, 2, 3, 4]), (0, [5]), (1, [1])]
    assert list(lay.v_seqlens) == [32, 32, 48]
    assert list(lay.s_seqlens) == [68, 22, 58, 8, 88, 34]
    Hq = 8
    for v, (_, mem) in enumerate(lay.virtual):
        for m, b in enumerate(mem):
            assert lay.q_rows[v * R + m] == b
            for h in range(Hq):
                assert lay.a_rows[b * Hq + h] == (v * R + m) * Hq + h
    assert np.all(lay.q_rows[5:8] == -1)  # padding of the second virtual request
    # the suffix page table starts at the first page after the prefix
    assert np.array_equal(lay.s_page_table[1, :4], w.page_table[1, 3:7])
    assert np.array_equal(lay.v_page_table[2, :3], w.page_table[1, :3])


def test_causal_multi_token_rows_and_ungrouped_requests():
    w = _w([64, 80, 50], [[0, 1]], [32], T=2, Hq=4, Hkv=2)
    lay = shared_prefix_layout(w.seqlens, w.page_table, w.prefix_groups, w.prefix_lens, 16, 2, 4, 2)
    assert lay.rows_per_virtual == 4  # 16 // (G=2 * T=2)
    assert np.all(lay.a_rows[2 * 2 * 4:] == -1)  # request 2 has no prefix state
    assert list(lay.s_seqlens) == [32, 48, 50]
    assert list(lay.q_rows[:4]) == [0, 1, 2, 3]  # (b, t) rows of requests 0 and 1


def test_invalid_groups_are_rejected():
    w = _w([64, 64, 64], [[0, 1]], [32])
    with pytest.raises(ValueError, match="multiple"):
        shared_prefix_layout(w.seqlens, w.page_table, [[0, 1]], [30], 16, 1, 8, 2)
    with pytest.raises(ValueError, match="share"):
        shared_prefix_layout(w.seqlens, w.page_table, [[0, 2]], [32], 16, 1, 8, 2)
    with pytest.raises(ValueError, match="repeated"):
        shared_prefix_layout(w.seqlens, w.page_table, [[0, 0]], [32], 16, 1, 8, 2)
    with pytest.raises(ValueError, match="after its prefix"):
        shared_prefix_layout(w.seqlens, w.page_table, [[0, 1]], [64], 16, 1, 8, 2)
