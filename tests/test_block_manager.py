"""The library's host block manager (C++, pkv_bm_*), on CPU.

Pinned to the pages' worked examples ("PagedAttention: Mathematical
Foundations ..." §4 block-table diagram, §5 copy-on-write diagram), to the
allocation lifecycle invariants of §4, and to the Python block-manager
fixture used by the workload generator (differential test on random
operation sequences).
"""
import numpy as np
import pytest

from paged_kv_cache_87_gb300 import binding, build, inputs
from tests.helpers import ints, read_golden


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def test_block_table_worked_example():
    g = read_golden("block_table_example.txt")
    B = int(g["block_size"])
    table = ints(g["table"])
    m = binding.BlockManager(32, B, free_order=table + [b for b in range(32) if b not in table])
    m.add_sequence(7, int(g["num_tokens"]))
    got, n = m.sequence(7)
    assert got == table and n == int(g["num_tokens"])
    # the next token (the 11th) goes to slot 19*4 + 2; a new block only after 12
    slot, cow = m.append_slot(7)
    assert slot == 19 * B + 2 and cow is None
    assert m.num_free == 32 - 3


def test_copy_on_write_worked_example():
    g = read_golden("cow_example.txt")
    B = int(g["block_size"])
    m = binding.BlockManager(16, B, free_order=[7, 1, 3] + [b for b in range(16)
                                                          if b not in (7, 1, 3)])
    m.add_sequence(1, int(g["prompt_tokens"]))
    m.fork(1, 2)
    assert [m.refcount(b) for b in ints(g["prompt_table"])] == ints(g["refcount_after_fork"])
    slot, cow = m.append_slot(1)              # sample 1 writes into shared block 1
    assert list(cow) == ints(g["cow_pair"])
    assert slot == 3 * B + int(g["prompt_tokens"]) % B
    assert m.sequence(1)[0] == ints(g["sample1_table"])
    assert m.sequence(2)[0] == ints(g["sample2_table"])
    for b in (7, 1, 3):
        assert m.refcount(b) == int(g[f"refcount_{b}"])
    slot2, cow2 = m.append_slot(2)             # sample 2 now owns block 1 alone
    assert cow2 is None and slot2 == 1 * B + int(g["prompt_tokens"]) % B


def test_lifecycle_invariants_and_free_order():
    B, NB = 16, 40
    m = binding.BlockManager(NB, B)
    m.add_sequence(0, 33)                     # 3 blocks
    assert m.sequence(0) == ([0, 1, 2], 33)
    for _ in range(15):                       # fills block 2 (48 tokens)
        assert m.append_slot(0)[1] is None
    assert m.sequence(0)[1] == 48 and len(m.sequence(0)[0]) == 3
    m.append_slot(0)                          # overflow -> block 3
    assert m.sequence(0)[0] == [0, 1, 2, 3]
    m.fork(0, 1)
    m.free_sequence(0)
    assert m.num_free == NB - 4 and all(m.refcount(b) == 1 for b in range(4))
    m.free_sequence(1)                        # freed blocks go to the back of the free list
    assert m.num_free == NB
    m.add_sequence(2, (NB - 4) * B)
    assert m.sequence(2)[0] == list(range(4, NB))


def test_errors_leave_state_unchanged():
    m = binding.BlockManager(4, 8)
    m.add_sequence(0, 24)
    with pytest.raises(binding.PagedKVError) as e:
        m.add_sequence(1, 17)
    assert e.value.status == binding.PKV_ERR_OUT_OF_BLOCKS
    m.fork(0, 1)
    m.fork(0, 2)
    # three appends: 0 overflows (needs a block), 1 and 2 too -> only one block left
    with pytest.raises(binding.PagedKVError):
        m.prepare_step([0, 1, 2], 8)
    assert m.num_free == 1 and m.sequence(0)[1] == 24 and m.refcount(0) == 3
    with pytest.raises(binding.PagedKVError):
        m.fork(0, 1)                          # id in use
    with pytest.raises(binding.PagedKVError):
        m.append_slot(99)


@pytest.mark.parametrize("seed", range(6))
def test_matches_python_fixture_on_random_operations(seed):
    """Same operations on the C++ manager and the generator's fixture give the same state."""
    rng = np.random.default_rng(seed)
    B, NB = int(rng.choice([8, 16, 32])), 200
    order = rng.permutation(NB)
    cpp = binding.BlockManager(NB, B, free_order=order)
    py = inputs.BlockManager(NB, B, rng=None, guards=False)
    py.free = [int(b) for b in order]
    tables, lens, next_id = {}, {}, 0
    for _ in range(300):
        op = rng.integers(0, 4) if tables else 0
        try:
            if op == 0:                                   # prefill
                n = int(rng.integers(1, 5 * B))
                if -(-n // B) > len(py.free):
                    continue
                cpp.add_sequence(next_id, n)
                tables[next_id], lens[next_id] = py.allocate(n), n
                next_id += 1
            elif op == 1:                                 # fork
                parent = int(rng.choice(list(tables)))
                cpp.fork(parent, next_id)
                tables[next_id], lens[next_id] = py.fork(tables[parent]), lens[parent]
                next_id += 1
            elif op == 2:                                 # append one token
                sid = int(rng.choice(list(tables)))
                t, n = tables[sid], lens[sid]
                need = n // B >= len(t) or py.refcount[t[n // B]] > 1
                if need and not py.free:
                    continue
                slot, cow = cpp.append_slot(sid)
                pair = None
                if n // B < len(t):
                    pair = py.copy_on_write(t, n // B)
                ref_slot = py.append_slot(t, n)
                lens[sid] = n + 1
                assert slot == ref_slot and cow == pair
            else:                                         # completion / pruning
                sid = int(rng.choice(list(tables)))
                cpp.free_sequence(sid)
                py.free_table(tables.pop(sid))
                lens.pop(sid)
        except binding.PagedKVError:
            raise
        for sid in tables:
            assert cpp.sequence(sid) == (tables[sid], lens[sid])
        assert cpp.num_free == len(py.free)
        for b in range(NB):
            assert cpp.refcount(b) == py.refcount[b]
        # §4: waste only in the last block of each sequence
        for sid, t in tables.items():
            assert 0 <= len(t) * B - lens[sid] <= B - 1


def test_prepare_step_batches_appends_and_cow():
    B = 16
    m = binding.BlockManager(64, B)
    m.add_sequence(0, 40)                  # 3 blocks, last partial
    for c in (1, 2, 3):
        m.fork(0, c)
    slots, pairs, tables, ctx = m.prepare_step([0, 1, 2, 3], 8)
    # the first three writers copy the shared partial block; the last keeps it
    assert len(pairs) == 3 and all(p[0] == 2 for p in pairs)
    assert len(set(pairs[:, 1].tolist())) == 3 and 2 not in pairs[:, 1]
    assert (ctx == 41).all()
    assert tables[3, 2] == 2 and slots[3] == 2 * B + 40 % B
    assert sorted(tables[:3, 2].tolist()) == sorted(pairs[:, 1].tolist())
    assert (tables[:, :2] == [0, 1]).all() and (tables[:, 3:] == -1).all()
    binding.validate_pairs(pairs, 64)


def test_prepare_step_needs_only_the_copies_it_makes():
    """Two sequences share a partial last block (refcount 2) and one block is free: the
    first writer copies it, the second becomes its sole owner, so the step fits."""
    B = 16
    m = binding.BlockManager(3, B)
    m.add_sequence(0, 20)                  # blocks 0, 1 (the second partial)
    m.fork(0, 1)
    assert m.num_free == 1
    slots, pairs, tables, ctx = m.prepare_step([0, 1], 4)
    assert len(pairs) == 1 and pairs[0][0] == 1 and pairs[0][1] == 2
    assert m.num_free == 0 and m.refcount(1) == 1 and m.refcount(2) == 1
    assert (ctx == 21).all()
    # three sharers of one block and a single free block: two copies are needed
    m2 = binding.BlockManager(4, B)
    m2.add_sequence(0, 20)
    m2.fork(0, 1)
    m2.fork(0, 2)
    assert m2.num_free == 2
    before = [m2.refcount(b) for b in range(4)]
    slots, pairs, tables, ctx = m2.prepare_step([0, 1, 2], 4)
    assert len(pairs) == 2 and m2.num_free == 0
    m3 = binding.BlockManager(3 + 1, B)
    m3.add_sequence(0, 20)
    m3.fork(0, 1)
    m3.fork(0, 2)
    m3.add_sequence(9, 1)                  # takes one of the two free blocks
    assert m3.num_free == 1
    before = [m3.refcount(b) for b in range(4)]
    with pytest.raises(binding.PagedKVError):
        m3.prepare_step([0, 1, 2], 4)      # two copies, one free block: refused
    assert [m3.refcount(b) for b in range(4)] == before and m3.num_free == 1


def _beam_invariants(m, live, NB):
    """Every block's reference count is the number of live beams whose table holds it;
    the free count is what no live beam holds."""
    held = {}
    for s in live:
        table, _ = m.sequence(s)
        for b in table:
            held[b] = held.get(b, 0) + 1
    for b in range(NB):
        assert m.refcount(b) == held.get(b, 0), b
    assert m.num_free == NB - len(held)
    return held


def test_beam_search_prunes_and_forks_by_reference_counts():
    """Beam search ("...Mathematical Foundations" §5 Beam Search): each step every live
    beam appends a token, then K survivors are forked from chosen parents and the old
    beams dropped. Only block tables and reference counts change: survivors share the
    parents' blocks, discarded beams give theirs back, and copy-on-write copies happen
    only where a shared block is written."""
    B, NB, K, prompt = 4, 128, 4, 10
    rng = np.random.default_rng(7)
    m = binding.BlockManager(NB, B)
    m.add_sequence(0, prompt)
    live, next_id = [0], 1
    for c in range(1, K):                     # the first K beams fork the prompt
        m.fork(0, c)
        live.append(c)
    next_id = K
    tokens = {s: prompt for s in live}
    copies = 0
    for step in range(12):
        slots, pairs, tables, ctx = m.prepare_step(live, 16)
        copies += len(pairs)
        for i, s in enumerate(live):
            tokens[s] += 1
            assert ctx[i] == tokens[s]
            assert slots[i] == tables[i][(tokens[s] - 1) // B] * B + (tokens[s] - 1) % B
        # every copy's destination is a fresh block held by exactly one beam
        for _, dst in pairs:
            assert m.refcount(int(dst)) == 1
        _beam_invariants(m, live, NB)
        # selection: K new beams, each a fork of a parent drawn from the live ones
        # (some parents several times, some not at all), then the old beams go
        parents = rng.choice(live, size=K, replace=True)
        new = []
        for par in parents:
            m.fork(int(par), next_id)
            tokens[next_id] = tokens[int(par)]
            new.append(next_id)
            next_id += 1
        for s in live:
            m.free_sequence(s)
        live = new
        held = _beam_invariants(m, live, NB)
        # survivors share history: fewer blocks than K private copies would take
        assert len(held) < K * -(-max(tokens[s] for s in live) // B)
    assert copies > 0
    for s in live:
        m.free_sequence(s)
    assert m.num_free == NB and all(m.refcount(b) == 0 for b in range(NB))
