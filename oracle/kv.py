"""Paged KV block tables: remap by ancestors, then append tokens (CPU oracle).

Test infrastructure: part of the CPU oracle (see ``oracle/__init__.py``).

"Faster LLM Inference via Sequential Monte Carlo" (gist.science explainer, zh:
section 2 "系统优化设计", KV Cache 优化; es: "Ventajas Sistémicas", Gestión de
Caché) says the resampling step manages the KV cache only by exchanging
pointers and updating reference counts, with no copy of KV data, and that
particles share their common prefix.  The pages give no data structure, so this
oracle takes the plainest paged-table reading:

  * each particle holds a table of T block ids and a token count L; block t
    holds tokens [t*bs, (t+1)*bs); entries past ceil(L/bs) are -1;
  * each prompt b owns a pool of P blocks with ids b*P .. b*P+P-1, a reference
    count per block (the number of table entries, over the prompt's particles,
    that name it) and a LIFO stack of free block ids;
  * remap (when the prompt resampled): particle i takes ancestor a_i's table
    and token count; every new reference adds 1, every old reference subtracts
    1; blocks whose count falls to 0 are pushed on the free stack in ascending
    id order;
  * append (every step): every particle grows by n tokens.  When n > 0, a
    partially filled tail block that several particles hold is kept by the
    lowest particle index; every other holder pops a fresh block and records a (src, dst)
    copy-on-write pair, the only KV data movement, which is left to the
    caller.  Further blocks needed for the new tokens are popped in
    ascending particle order, fork first.  Popped blocks get count 1.
  * if the pops of a prompt exceed its free stack, or a particle would need
    more than T blocks, the append of that prompt is skipped and an error is
    reported.
"""
import numpy as np

from .errors import (OracleError, DEV_POOL_EXHAUSTED, DEV_TABLE_OVERFLOW,
                     DEV_BAD_BLOCK)


def n_blocks(length, block_size):
    """Blocks needed to hold ``length`` tokens."""
    return (int(length) + block_size - 1) // block_size


def _check_ids(ids, b, pool):
    for blk in ids:
        if not (b * pool <= blk < (b + 1) * pool):
            raise OracleError(DEV_BAD_BLOCK, f"block {blk} outside prompt {b}'s pool")


def remap_append(tables, seq_len, refcount, free_list, free_top, ancestors,
                 resampled, n_append, block_size, pool):
    """Remap by ancestors (where resampled) and append ``n_append`` tokens.

    tables [B,N,T], seq_len [B,N], refcount [B*P], free_list [B,P],
    free_top [B], ancestors [B,N], resampled [B].  Inputs are not modified.

    Returns dict(tables, seq_len, refcount, free_list, free_top,
    cow_pairs: list of B lists of (src, dst), errors: list of B lists of
    error kinds).
    """
    tables = np.array(tables, dtype=np.int64)
    seq_len = np.array(seq_len, dtype=np.int64)
    refcount = np.array(refcount, dtype=np.int64)
    free_list = np.array(free_list, dtype=np.int64)
    free_top = np.array(free_top, dtype=np.int64)
    big_b, n_part, t_max = tables.shape
    cow_pairs = [[] for _ in range(big_b)]
    errors = [[] for _ in range(big_b)]
    for b in range(big_b):
        # ---- remap: pointer exchange and reference counts -------------------
        if resampled[b]:
            old_tables = tables[b].copy()
            old_len = seq_len[b].copy()
            a = np.asarray(ancestors[b], dtype=np.int64)
            old_refs = [int(old_tables[j, t]) for j in range(n_part)
                        for t in range(n_blocks(old_len[j], block_size))]
            _check_ids(old_refs, b, pool)
            for i in range(n_part):
                tables[b, i] = old_tables[a[i]]
                seq_len[b, i] = old_len[a[i]]
                for t in range(n_blocks(old_len[a[i]], block_size)):
                    refcount[old_tables[a[i], t]] += 1
            for blk in old_refs:
                refcount[blk] -= 1
            freed = sorted({blk for blk in old_refs if refcount[blk] == 0})
            for blk in freed:
                free_list[b, free_top[b]] = blk
                free_top[b] += 1
        # ---- append: copy-on-write of shared partial tails, then growth -----
        tails = []
        for i in range(n_part):
            length = int(seq_len[b, i])
            if length % block_size:
                tails.append(int(tables[b, i, n_blocks(length, block_size) - 1]))
            else:
                tails.append(None)
        # a shared partial tail is forked only when tokens will be written into it
        forks = [n_append > 0 and tails[i] is not None and tails[i] in tails[:i]
                 for i in range(n_part)]
        grows = [n_blocks(seq_len[b, i] + n_append, block_size) - n_blocks(seq_len[b, i], block_size)
                 for i in range(n_part)]
        if any(n_blocks(seq_len[b, i] + n_append, block_size) > t_max for i in range(n_part)):
            errors[b].append(DEV_TABLE_OVERFLOW)
            continue
        if sum(forks) + sum(grows) > free_top[b]:
            errors[b].append(DEV_POOL_EXHAUSTED)
            continue

        def pop():
            free_top[b] -= 1
            return int(free_list[b, free_top[b]])

        for i in range(n_part):
            length = int(seq_len[b, i])
            nb = n_blocks(length, block_size)
            if forks[i]:
                src = tails[i]
                dst = pop()
                cow_pairs[b].append((src, dst))
                tables[b, i, nb - 1] = dst
                refcount[dst] = 1
                refcount[src] -= 1
            for g in range(grows[i]):
                blk = pop()
                tables[b, i, nb + g] = blk
                refcount[blk] = 1
            seq_len[b, i] = length + n_append
    return dict(tables=tables, seq_len=seq_len, refcount=refcount,
                free_list=free_list, free_top=free_top, cow_pairs=cow_pairs,
                errors=errors)


def live_references(tables, seq_len, block_size):
    """Count of table references per block id (dict), for invariant checks."""
    counts = {}
    big_b, n_part, _ = np.shape(tables)
    for b in range(big_b):
        for i in range(n_part):
            for t in range(n_blocks(seq_len[b][i], block_size)):
                blk = int(tables[b][i][t])
                counts[blk] = counts.get(blk, 0) + 1
    return counts


def usage(tables, seq_len, block_size):
    """Blocks held with sharing against blocks N unshared copies would hold.

    Per prompt b: used[b] = number of distinct blocks its particles' tables
    reference; unshared[b] = sum over particles of the blocks each particle's
    tokens fill on their own.  The SMC page (section 2, "系统优化设计") credits
    prefix sharing and pointer exchange with a smaller KV cache; 1 -
    used/unshared is that saving for one state.
    """
    big_b, n_part, _ = np.shape(tables)
    used = np.zeros(big_b, dtype=np.int64)
    unshared = np.zeros(big_b, dtype=np.int64)
    for b in range(big_b):
        seen = set()
        for i in range(n_part):
            nb = n_blocks(seq_len[b][i], block_size)
            unshared[b] += nb
            for t in range(nb):
                seen.add(int(tables[b][i][t]))
        used[b] = len(seen)
    return used, unshared
