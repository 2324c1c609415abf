"""The roofline numerator: algorithmic bytes per step, counted from first
principles on small cases, and the figures quoted for the named workloads
(CPU only)."""
import workloads as W


def test_gqa_bytes_by_hand():
    # 2 requests of 20 and 33 tokens, 4 q / 2 kv heads, D = 16, pages of 16
    w = W.make_custom([20, 33], num_q_heads=4, num_kv_heads=2, head_dim_qk=16, page_size=16, seed=0)
    kv = (20 + 33) * 2 * (16 + 16) * 2          # K and V rows of both kv heads, bf16
    rows = 2 * 1 * 4                             # batch x T x Hq query rows
    q_out_lse = rows * 16 * 2 + rows * 16 * 2 + rows * 4
    pages = (2 + 3) * 4                          # ceil(20/16) + ceil(33/16) page-table entries
    assert w.algorithmic_bytes() == kv + q_out_lse + pages


def test_mla_bytes_by_hand():
    # one latent row of 576 values per token; V is its first 512 values (not read twice)
    w = W.make_custom([100, 64], mla=True, num_q_heads=4, head_dim_qk=576, head_dim_v=512, page_size=64,
                      seed=0)
    rows = 2 * 4
    expect = (164 * 576 * 2) + rows * 576 * 2 + rows * 512 * 2 + rows * 4 + (2 + 1) * 4
    assert w.algorithmic_bytes() == expect


def test_sparse_and_shared_prefix_bytes():
    base = W.make_custom([300, 200, 50], mla=True, num_q_heads=2, head_dim_qk=576, head_dim_v=512,
                         page_size=64, seed=1)
    s = W.select_topk(base, 64)
    listed = 64 + 64 + 50
    rows = 3 * 2
    # each listed row: the latent row, one page-table entry and one index
    assert s.algorithmic_bytes() == listed * 576 * 2 + rows * (576 + 512) * 2 + rows * 4 + 2 * listed * 4
    g = W.make_custom([4096 + 100, 4096 + 7, 900], num_q_heads=8, num_kv_heads=2, head_dim_qk=64,
                      page_size=16, seed=2)
    p = W.share_prefix(g, [[0, 1]], [4096])
    # the shared 4096 tokens (256 pages) are counted once
    assert p.kv_tokens == g.kv_tokens - 4096
    assert p.algorithmic_bytes() == g.algorithmic_bytes() - 4096 * 2 * 128 * 2 - 256 * 4


def test_named_workload_figures():
    # the per-step bytes quoted next to the measurements
    assert W.make("llama3_8b_gqa").algorithmic_bytes() == 598_183_620
    assert W.make("mla_absorbed").algorithmic_bytes() == 670_750_944
    assert W.make("mla_sparse_top2048").algorithmic_bytes() == 163_208_880
    assert W.make("shared_prefix_gqa").algorithmic_bytes() == 209_465_864
