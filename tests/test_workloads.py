"""The seeded input recipe (paged_kv_extend_gb300/workloads.py), which feeds
both the oracle and the CUDA path: determinism, the slot permutation, the
index arrays it hands out, the pool it scatters, the length distributions of
the named workloads, the MLA aliasing and the draft-tree mask."""
import dataclasses

import torch

from paged_kv_extend_gb300 import workloads as W


def _cheap(name):
    """The named workload's lengths and slots with tiny heads (lengths and the
    slot permutation are drawn before any value, so they are the same)."""
    return dataclasses.replace(W.SPECS[name], hq=1, hkv=1, lq=8, lv=8, v_aliases_k=False)


def test_same_seed_same_workload():
    a, b = W.draw(W.SPECS["tiny"]), W.draw(W.SPECS["tiny"])
    for f in ("slots", "k_rows", "v_rows", "q", "kv_indices", "extend_kv_indices"):
        assert torch.equal(getattr(a, f), getattr(b, f)), f
    c = W.draw(W.SPECS["tiny"], seed=5)
    assert not torch.equal(a.q, c.q)


def test_slots_are_distinct_pool_rows_and_index_arrays_follow_them():
    spec = W.small_spec(batch=4, prefix=[5, 0, 130, 17], extend=[3, 17, 1, 40], seed=11)
    wl = W.draw(spec)
    T = [p + e for p, e in zip(wl.prefix_lens, wl.extend_lens)]
    slots = wl.slots.tolist()
    assert len(slots) == sum(T) and len(set(slots)) == len(slots)
    assert min(slots) >= 0 and max(slots) < spec.num_slots
    pre, ext, off = [], [], 0
    for b, t in enumerate(T):
        pre += slots[off: off + wl.prefix_lens[b]]
        ext += slots[off + wl.prefix_lens[b]: off + t]
        off += t
    assert wl.kv_indices.tolist() == pre and wl.extend_kv_indices.tolist() == ext
    assert wl.kv_indptr.tolist() == [0, 5, 5, 135, 152]
    assert wl.qo_indptr.tolist() == [0, 3, 20, 21, 61]
    assert wl.extend_seq_lens.tolist() == wl.extend_lens
    starts = wl.extend_start_loc.tolist()
    for b in range(4):  # each sequence's extend slots start at its extend_start_loc
        assert ext[starts[b]: starts[b] + wl.extend_lens[b]] == slots[
            int(wl.token_offsets[b]) + wl.prefix_lens[b]: int(wl.token_offsets[b]) + T[b]]


def test_pool_holds_every_token_row_at_its_slot_and_zeros_elsewhere():
    wl = W.draw(W.small_spec(batch=2, prefix=[9, 4], extend=[2, 6], seed=3))
    kb, vb = wl.pool()
    s = wl.slots.to(torch.int64)
    assert torch.equal(kb[s], wl.k_rows) and torch.equal(vb[s], wl.v_rows)
    other = torch.ones(kb.shape[0], dtype=torch.bool)
    other[s] = False
    assert kb[other].abs().sum() == 0 and vb[other].abs().sum() == 0
    k_ext, v_ext = wl.extend_kv()
    rows = wl.extend_rows()
    assert torch.equal(k_ext, wl.k_rows[rows]) and torch.equal(v_ext, wl.v_rows[rows])


def test_named_workload_lengths_follow_their_distributions():
    l8 = W.draw(_cheap("llama3_8b"))
    assert all(0 <= p <= 4096 for p in l8.prefix_lens)
    assert all(1 <= e <= 1024 for e in l8.extend_lens)
    lp = W.draw(_cheap("long_prefix"))
    assert set(lp.prefix_lens) == {8192} and set(lp.extend_lens) == {16}
    ht = W.draw(_cheap("heavy_tail"))
    assert all(0 <= p <= 16384 for p in ht.prefix_lens)
    assert all(1 <= e <= 4096 for e in ht.extend_lens)
    assert max(ht.extend_lens) > 8 * sorted(ht.extend_lens)[len(ht.extend_lens) // 2]  # heavy tail
    dg = W.draw(_cheap("decode_gqa"))
    assert dg.q.shape[0] == dg.batch and dg.kv_indptr.tolist()[-1] == dg.batch * 8193


def test_mla_values_are_the_first_512_dims_of_the_key_rows():
    spec = W.small_spec(batch=2, hq=16, hkv=1, lq=576, lv=512, prefix=[3, 0], extend=[2, 4],
                        v_aliases_k=True, std=0.5, seed=4)
    wl = W.draw(spec)
    assert torch.equal(wl.v_rows, wl.k_rows[..., :512])
    kb, vb = wl.pool()
    assert torch.equal(vb, kb[..., :512])


def test_draft_tree_mask_rows_see_prefix_ancestors_and_self():
    spec = dataclasses.replace(W.SPECS["spec_verify"], batch=2, hq=1, hkv=1, lq=8, lv=8,
                               prefix=[5, 0], extend=[6, 3], num_slots=64)
    wl = W.draw(spec)
    for b in range(2):
        P, E = wl.prefix_lens[b], wl.extend_lens[b]
        rows = wl.custom_mask[int(wl.mask_indptr[b]): int(wl.mask_indptr[b + 1])].view(E, P + E)
        assert rows[:, :P].all()                       # every node sees the whole prefix
        assert rows[:, P:].diagonal().all()            # and itself
        assert not rows[:, P:].triu(1).any()           # never a later node
        assert rows[1:, P].all() if E > 1 else True    # node 0 is every node's ancestor
