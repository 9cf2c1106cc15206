"""Pins of the oracle's block-table remap and append (CPU only).

A shadow KV store holds one token id per slot.  Each step replays what a
serving engine would do with the oracle's outputs: copy every copy-on-write
block, then write the appended tokens through the new tables.  Every particle's
sequence read back through its table must equal the sequence tracked directly
from the ancestors, which fails if a shared block is ever written, a fork is
missed or a table entry points at the wrong block.
"""
import numpy as np
import pytest

from oracle import kv, smc
from oracle.errors import DEV_POOL_EXHAUSTED, DEV_TABLE_OVERFLOW, DEV_BAD_BLOCK, OracleError
from smc_speculative_decoding_gb300.workloads import make_kv_state


def _state(big_b, n, prefix, bs, t_len, pool):
    s = make_kv_state(big_b, n, prefix, bs, t_len, pool)
    return {k: v.numpy().astype(np.int64) for k, v in s.items()}


def _check_invariants(st, big_b, n, bs, pool):
    refs = kv.live_references(st["tables"], st["seq_len"], bs)
    for b in range(big_b):
        free = list(st["free_list"][b, :st["free_top"][b]])
        assert len(free) == len(set(free)), "block pushed twice"
        for blk in range(b * pool, (b + 1) * pool):
            assert st["refcount"][blk] == refs.get(blk, 0)
            assert (blk in free) == (refs.get(blk, 0) == 0), f"block {blk} leaked or double-owned"
        tails = [st["tables"][b, i, kv.n_blocks(st["seq_len"][b, i], bs) - 1]
                 for i in range(n) if st["seq_len"][b, i] % bs]
        assert len(tails) == len(set(tails)), "partial tail shared after append"
        for i in range(n):
            nb = kv.n_blocks(st["seq_len"][b, i], bs)
            assert (st["tables"][b, i, nb:] == -1).all()


@pytest.mark.parametrize("prefix,bs", [(10, 4), (16, 4), (5, 16), (0, 4)])
def test_shadow_store_replay(prefix, bs):
    big_b, n, n_app, steps = 2, 6, 3, 8
    t_len = kv.n_blocks(prefix + steps * n_app, bs) + 1
    pool = n * t_len
    st = _state(big_b, n, prefix, bs, t_len, pool)
    store = np.full((big_b * pool, bs), -1, dtype=np.int64)
    seqs = [[list(range(1000, 1000 + prefix)) for _ in range(n)] for _ in range(big_b)]
    for b in range(big_b):
        for pos in range(prefix):
            store[st["tables"][b, 0, pos // bs], pos % bs] = 1000 + pos
    rng = np.random.default_rng(prefix * 31 + bs)
    next_tok = 0
    for step in range(steps):
        resampled = rng.random(big_b) < 0.6
        anc = np.zeros((big_b, n), dtype=np.int64)
        for b in range(big_b):
            w = rng.dirichlet(np.full(n, 0.3))
            anc[b] = smc.systematic_resample(w, rng.random())[0] if resampled[b] else np.arange(n)
        out = kv.remap_append(st["tables"], st["seq_len"], st["refcount"], st["free_list"],
                              st["free_top"], anc, resampled, n_app, bs, pool)
        assert all(not e for e in out["errors"])
        for b in range(big_b):
            for src, dst in out["cow_pairs"][b]:
                store[dst] = store[src]
            seqs[b] = [list(seqs[b][a]) for a in anc[b]]
            for i in range(n):
                length = len(seqs[b][i])
                assert out["seq_len"][b, i] == length + n_app
                for pos in range(length, length + n_app):
                    blk = out["tables"][b, i, pos // bs]
                    assert out["refcount"][blk] == 1, "writing into a shared block"
                    store[blk, pos % bs] = next_tok
                    seqs[b][i].append(next_tok)
                    next_tok += 1
        st = {k: out[k] for k in ("tables", "seq_len", "refcount", "free_list", "free_top")}
        _check_invariants(st, big_b, n, bs, pool)
        for b in range(big_b):
            for i in range(n):
                length = st["seq_len"][b, i]
                got = [store[st["tables"][b, i, pos // bs], pos % bs] for pos in range(length)]
                assert got == seqs[b][i]


def test_remap_is_pointer_exchange_only():
    """With no append the only change is to tables, counts and the free stack."""
    big_b, n, bs, prefix = 1, 4, 4, 9
    st = _state(big_b, n, prefix, bs, 8, 32)
    first = kv.remap_append(st["tables"], st["seq_len"], st["refcount"], st["free_list"],
                            st["free_top"], np.tile(np.arange(n), (1, 1)), [False], 4, bs, 32)
    anc = np.array([[2, 2, 2, 0]])
    out = kv.remap_append(first["tables"], first["seq_len"], first["refcount"],
                          first["free_list"], first["free_top"], anc, [True], 0, bs, 32)
    assert out["cow_pairs"] == [[]]
    for i, a in enumerate(anc[0]):
        assert np.array_equal(out["tables"][0, i], first["tables"][0, a])
    # particles 1 and 3 lost their private blocks: pushed in ascending id order
    freed = list(out["free_list"][0, first["free_top"][0]:out["free_top"][0]])
    assert freed == sorted(freed) and len(freed) == 2 * 2  # each held 2 private blocks


def test_pool_exhausted_and_table_overflow_skip_the_append():
    st = _state(1, 4, 16, 4, 6, 7)  # 4 prefix blocks, 3 free
    out = kv.remap_append(st["tables"], st["seq_len"], st["refcount"], st["free_list"],
                          st["free_top"], np.arange(4)[None], [False], 4, 4, 7)
    assert out["errors"] == [[DEV_POOL_EXHAUSTED]]
    assert np.array_equal(out["seq_len"], st["seq_len"])
    st = _state(1, 2, 16, 4, 5, 20)
    out = kv.remap_append(st["tables"], st["seq_len"], st["refcount"], st["free_list"],
                          st["free_top"], np.arange(2)[None], [False], 5, 4, 20)
    assert out["errors"] == [[DEV_TABLE_OVERFLOW]]


def test_block_outside_pool_is_rejected():
    st = _state(2, 2, 8, 4, 4, 8)
    st["tables"][1, 0, 0] = 3  # prompt 0's block
    with pytest.raises(OracleError) as e:
        kv.remap_append(st["tables"], st["seq_len"], st["refcount"], st["free_list"],
                        st["free_top"], np.array([[0, 0], [1, 1]]), [True, True], 1, 4, 8)
    assert e.value.kind == DEV_BAD_BLOCK
