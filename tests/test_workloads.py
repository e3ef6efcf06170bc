"""The seeded input generator (no GPU): the same seed gives the same tensors, the shapes
and lengths of the named workloads are what their descriptions say, and the block table is
a permutation of the pool."""
import numpy as np
import torch

from query_aware_kv_gb300 import workloads as wl


def _small(seed):
    return wl.build("w", batch=3, num_q_heads=8, num_kv_heads=4, page_size=16,
                    prefill_lens=[100, 0, 33], steps=2, budget=64, seed=seed, outliers=2)


def test_same_seed_same_inputs_other_seed_other_inputs():
    a, b, c = _small(1), _small(1), _small(2)
    for name in ("k_pool", "v_pool", "block_table", "q", "k_new", "v_new"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    assert not torch.equal(a.k_pool, c.k_pool)


def test_block_table_is_a_permutation_of_the_pool():
    w = _small(3)
    pages = [wl.pages_for(int(L) + w.steps, w.page_size) for L in w.seq_lens.tolist()]
    used = np.concatenate([w.block_table[b, :n].numpy() for b, n in enumerate(pages)])
    assert sorted(used.tolist()) == list(range(w.num_phys))
    for b, n in enumerate(pages):
        assert (w.block_table[b, n:] == -1).all()


def test_named_workload_shapes():
    t = wl.tiny(seed=0)
    assert (t.batch, t.num_q_heads, t.num_kv_heads, t.page_size, t.top_k) == (1, 4, 4, 16, 16)
    assert int(t.seq_lens[0]) + t.steps == 1024
    lc = wl.longchat_32k(seed=0, steps=2)
    assert (lc.num_q_heads, lc.num_kv_heads, lc.top_k) == (32, 32, 128)
    assert int(lc.seq_lens[0]) == 32768
    assert len(lc.needles) == 8 * 32
    # every needle key is the fixed 4 sqrt(d) unit direction of its head's query
    b, g, p, slot = lc.needles[0]
    phys = int(lc.block_table[b, p])
    key = lc.k_pool[phys, g, slot].float()
    assert abs(float(key.norm()) - 4.0 * 128 ** 0.5) < 0.1


def test_outlier_channels_are_scaled():
    w = _small(4)
    assert w.outlier_channels.shape == (4, 2)
    g = 0
    ch = w.outlier_channels[g]
    other = [i for i in range(128) if i not in ch.tolist()]
    big = w.k_pool[:, g, :, ch].float().abs().mean()
    small = w.k_pool[:, g, :, other].float().abs().mean()
    assert big > 4 * small
