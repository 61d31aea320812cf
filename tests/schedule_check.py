"""Check a native schedule by invariants, from the device tables themselves.

``tree_attn_plan_describe_schedule`` prints the tables a run's kernels read:
work units, each CTA's unit range, blocks (page, span position * 32 + valid
slots, phase bit 30), row records (token, visible end, first partial slot,
partial count | (slot + 1) << 24), merge items and each token's first partial
slot.  ``check_schedule`` decodes them the way the kernels do and asserts:

* every (query token, q head) attends to exactly the keys of its path (its
  ancestors in full, then its own node up to its visible end: DeFT notes page,
  "Tree attention definition"), each key once, across all the units that
  carry its rows;
* the row's results land in exactly one place per partial: the output when
  the token has one partial, else each of its partial slots exactly once
  (the slots of the log-sum-exp merge, DeFT notes page, "Tree-Topology-Aware
  Global Reduction Strategy"), and every key of a slot's row sits in that
  slot's unit;
* a unit reads the key of a page only through that page's own kv head
  (grouped-query attention: q head h reads kv head h // (Hq / Hkv));
* the CTA ranges cover every unit exactly once and the merge items are the
  tokens with two or more partials, with disjoint partial ranges;
* a unit carries the read-once flag exactly when no other unit reads any
  (page, kv head) it reads (zero-valid filler pages aside), and the plan
  asks for L2 policies exactly when flagged units hold 3/4 of the tiles.

Keys are compared as multisets through a count and a sum of random 64-bit
hashes per (token, q head): a dropped, doubled or foreign key changes the sum
unless a 2^-64 accident hides it.  This is test code: it decodes tables, it
computes no attention and shares nothing with the kernels or the oracle.
"""
from __future__ import annotations

import numpy as np

PATH_MMA, PATH_HEADS, PATH_PHASES, PATH_PAIRS, PATH_READ_ONCE = 1, 2, 4, 16, 32
PHASE_SHIFT = 30
POS_MASK = (1 << PHASE_SHIFT) - 1
MMA_TILE_ROWS, SIMT_TILE_ROWS, SLOT_ROWS, PAIR_ROWS, BLOCKS_PER_TILE = 128, 8, 32, 64, 4


def _key_tables(spec, seed=12345):
    """Random hash per (page, kv head, slot), and its prefix sums over slots."""
    rng = np.random.default_rng(seed)
    h = rng.integers(0, 2**63, size=(spec.num_pages, spec.n_kv_heads, 16), dtype=np.uint64)
    h = h * np.uint64(2) + rng.integers(0, 2, size=h.shape, dtype=np.uint64)
    pre = np.zeros((spec.num_pages, spec.n_kv_heads, 17), dtype=np.uint64)
    pre[:, :, 1:] = np.cumsum(h, axis=2, dtype=np.uint64)
    return pre


def expected_keys(spec, pre):
    """Count and hash sum of each query token's path keys, per kv head."""
    nq, hkv = spec.n_queries, spec.n_kv_heads
    cnt = np.zeros(nq, dtype=np.int64)
    hs = np.zeros((nq, hkv), dtype=np.uint64)
    node_sum = {}

    def node_hash(a, n):
        key = (a, n)
        if key not in node_sum:
            p0 = int(spec.node_page_offsets[a])
            tot = np.zeros(hkv, dtype=np.uint64)
            for i in range((n + 15) // 16):
                tot += pre[int(spec.node_pages[p0 + i]), :, min(16, n - 16 * i)]
            node_sum[key] = tot
        return node_sum[key]

    for t in range(nq):
        u = int(spec.query_node[t])
        e = int(spec.query_kv_end[t])
        tot = node_hash(u, e).copy()
        c = e
        x = int(spec.parent[u])
        while x >= 0:
            n = int(spec.node_kv_len[x])
            tot += node_hash(x, n)
            c += n
            x = int(spec.parent[x])
        cnt[t] = c
        hs[t] = tot
    return cnt, hs


def decode(sched):
    units = np.asarray(sched["units"], dtype=np.int64).reshape(-1, 8)
    blocks = np.asarray(sched["blocks"], dtype=np.int64).reshape(-1, 2)
    rows = np.asarray(sched["rows"], dtype=np.int64).reshape(-1, 4)
    merge = np.asarray(sched["merge"], dtype=np.int64).reshape(-1, 4)
    return units, blocks, rows, merge


def unit_kind(u, rec_slot):
    """A label for what kind of unit this is (for choosing test tokens)."""
    tok_off, kvh, row0, nrows, b0, b1, chunk, path = (int(x) for x in u)
    if not path & PATH_MMA:
        return "simt"
    if path & PATH_PAIRS:
        return "pairs"
    if path & PATH_PHASES:
        return "packed_phases"
    if path & PATH_HEADS:
        return "packed_heads"
    if rec_slot >= 0:
        return "packed"
    return "mma_full" if nrows > 64 else "mma_half"


def check_schedule(spec, sched, num_sms=None, collect=False):
    """Assert the invariants above; with ``collect``, return per-token facts:
    the unit kinds its rows run in and whether a row of it is masked inside a
    tile (a causal tail or a node end inside the tile)."""
    hq, hkv, r = spec.n_q_heads, spec.n_kv_heads, spec.gqa
    assert sched["hq"] == hq and sched["hkv"] == hkv and sched["gqa"] == r
    units, blocks, rows, merge = decode(sched)
    poff = np.asarray(sched["poff"], dtype=np.int64)
    nq = spec.n_queries
    npart = int(sched["n_partials"])
    pre = _key_tables(spec)
    exp_cnt, exp_hash = expected_keys(spec, pre)

    # ---- CTA ranges
    cta = np.asarray(sched["cta_off"], dtype=np.int64)
    assert cta[0] == 0 and cta[-1] == len(units) and np.all(np.diff(cta) >= 0)
    assert len(cta) - 1 == sched["grid"]
    if num_sms is not None and len(units):
        assert sched["grid"] <= 2 * num_sms

    # ---- pages referenced
    if len(blocks):
        assert blocks[:, 0].min() >= 0 and blocks[:, 0].max() < spec.num_pages

    pcount = np.zeros(nq, dtype=np.int64)
    for rec in rows:
        if rec[0] >= 0:
            pcount[rec[0]] = rec[3] & 0xFFFFFF

    out_w = np.zeros((nq, hq), dtype=np.int64)
    out_c = np.zeros((nq, hq), dtype=np.int64)
    out_h = np.zeros((nq, hq), dtype=np.uint64)
    part_w = np.zeros((max(npart, 1), hq), dtype=np.int64)
    part_c = np.zeros((max(npart, 1), hq), dtype=np.int64)
    part_h = np.zeros((max(npart, 1), hq), dtype=np.uint64)
    part_tok = np.full(max(npart, 1), -1, dtype=np.int64)
    kinds = [set() for _ in range(nq)] if collect else None
    masked = np.zeros(nq, dtype=bool)

    for u in units:
        tok_off, kvh, row0, nrows, b0, b1, chunk, path = (int(x) for x in u)
        mma = bool(path & PATH_MMA)
        nr = min(nrows, MMA_TILE_ROWS if mma else SIMT_TILE_ROWS)
        if nr <= 0:
            continue
        i = np.arange(nr)
        grow = row0 + i
        rec = rows[tok_off + grow // r]
        tok, vis, pbase, pcs = rec[:, 0], rec[:, 1], rec[:, 2], rec[:, 3]
        slot = (pcs >> 24) - 1
        live = tok >= 0
        if not live.any():
            continue
        # q head of each row (a unit packed by kv head: 32-row slot k is kv head
        # kvh + k; a pair unit: 64-row slot k)
        pairs = bool(mma and path & PATH_PAIRS)
        head_kv = kvh + (grow // SLOT_ROWS if (mma and path & PATH_HEADS)
                         else grow // PAIR_ROWS if pairs else 0)
        head = head_kv * r + grow % r
        # blocks of the unit, tile by tile: page index bb inside its tile
        nb = b1 - b0
        bi = np.arange(nb)
        bb = bi % BLOCKS_PER_TILE
        page = blocks[b0:b1, 0]
        meta = blocks[b0:b1, 1]
        valid = meta & 31
        if mma and pairs:
            # a pair unit: the rows of 64-row slot k see pages 2k, 2k + 1 of each tile
            k = i // PAIR_ROWS
            assert np.all(~live | (slot == k)), "pair row outside its slot"
            see = (bb[None, :] // 2) == k[:, None]
            pos = np.broadcast_to(meta[None, :] >> 5, (nr, nb))
        elif mma:
            warp = i // 32
            packed = slot >= 0
            # a packed row reads page `warp` of each tile only; the planner
            # puts slot k's rows in warp k
            assert np.all(~(packed & live) | (slot == warp)), "packed row outside its warp"
            pos_all = meta >> 5  # non-packed rows: span position (no phase bit expected)
            pos_packed = (meta & POS_MASK) >> 5
            see = np.where(packed[:, None], bb[None, :] == warp[:, None], True)
            if path & PATH_PHASES:
                phase = (meta >> PHASE_SHIFT) & 1
                mine = (i % 32) >> 4
                see &= np.where(packed[:, None], phase[None, :] == mine[:, None], True)
            pos = np.where(packed[:, None], pos_packed[None, :], pos_all[None, :])
        else:
            packed = slot >= 0
            see = np.where(packed[:, None], bb[None, :] == slot[:, None], True)
            pos = np.broadcast_to(meta[None, :] >> 5, (nr, nb))
        lim = np.clip(np.minimum(valid[None, :], vis[:, None] - pos), 0, None)
        lim = np.where(see & live[:, None], lim, 0)
        # kv head whose K/V the block's page is loaded with
        blk_kv = kvh + (bb if (mma and path & PATH_HEADS) else bb // 2 if pairs else 0)
        bkv = np.broadcast_to(blk_kv, (nb,)) if np.ndim(blk_kv) else np.full(nb, blk_kv)
        used = lim > 0
        if used.any():
            rr, cc = np.nonzero(used)
            assert np.all(bkv[cc] == head[rr] // r), "key from another kv head"
        cnt = lim.sum(axis=1)
        hsum = pre[page[None, :], bkv[None, :], lim].sum(axis=1, dtype=np.uint64) if nb else \
            np.zeros(nr, dtype=np.uint64)
        if collect:
            part_mask = (lim > 0) & (lim < valid[None, :])
            for k in np.nonzero(live)[0]:
                kinds[tok[k]].add(unit_kind(u, slot[k]))
                if part_mask[k].any():
                    masked[tok[k]] = True
        for k in np.nonzero(live)[0]:
            t, h = int(tok[k]), int(head[k])
            if pbase[k] < 0:
                out_w[t, h] += 1
                out_c[t, h] += cnt[k]
                out_h[t, h] += hsum[k]
            else:
                ps = int(pbase[k]) + chunk
                assert 0 <= ps < npart
                part_w[ps, h] += 1
                part_c[ps, h] += cnt[k]
                part_h[ps, h] += hsum[k]
                assert part_tok[ps] in (-1, t)
                part_tok[ps] = t

    # ---- read-once flags: (page, kv head) pairs read by exactly one unit
    def heads_of(u):
        kvh, b0, b1, path = int(u[1]), int(u[4]), int(u[5]), int(u[7])
        bb = np.arange(b1 - b0) % BLOCKS_PER_TILE
        mma = bool(path & PATH_MMA)
        if mma and path & PATH_HEADS:
            return kvh + bb
        if mma and path & PATH_PAIRS:
            return kvh + bb // 2
        return np.full(b1 - b0, kvh)
    keys = []
    for ui, u in enumerate(units):
        b0, b1 = int(u[4]), int(u[5])
        real = (blocks[b0:b1, 1] & 31) > 0
        k = blocks[b0:b1, 0].astype(np.int64) * hkv + heads_of(u)
        keys.append(k[real])
    allk = np.concatenate(keys) if keys else np.zeros(0, np.int64)
    uniq, counts = np.unique(allk, return_counts=True)
    cnt_of = dict(zip(uniq.tolist(), counts.tolist()))
    tiles = once_tiles = 0
    for u, k in zip(units, keys):
        once = int(u[5]) > int(u[4]) and all(cnt_of[int(x)] == 1 for x in k)
        assert bool(int(u[7]) & PATH_READ_ONCE) == once, "read-once flag"
        t = (int(u[5]) - int(u[4]) + BLOCKS_PER_TILE - 1) // BLOCKS_PER_TILE
        tiles += t
        once_tiles += t if once else 0
    if "kv_evict" in sched:
        assert bool(sched["kv_evict"]) == (tiles > 0 and 4 * once_tiles >= 3 * tiles), "kv_evict"

    # ---- merge items: tokens with >= 2 partials, disjoint slot ranges
    assert sorted(merge[:, 0].tolist()) == [t for t in range(nq) if pcount[t] >= 2]
    seen = np.zeros(max(npart, 1), dtype=np.int64)
    for tok, off, count, _ in merge:
        assert off == poff[tok] and count == pcount[tok]
        seen[off:off + count] += 1
    if npart:
        assert np.all(seen[:npart] == 1), "partial slots not a partition"

    # ---- every (token, q head): its keys exactly once, each result once
    for t in range(nq):
        kv = np.arange(hq) // r
        if pcount[t] <= 1:
            assert pcount[t] == 1, f"token {t} has no group"
            assert np.all(out_w[t] == 1), f"token {t}: output written {out_w[t]} times"
            assert np.all(out_c[t] == exp_cnt[t]), f"token {t}: key count"
            assert np.all(out_h[t] == exp_hash[t, kv]), f"token {t}: key set"
        else:
            assert np.all(out_w[t] == 0)
            sl = slice(int(poff[t]), int(poff[t] + pcount[t]))
            assert np.all(part_w[sl] == 1), f"token {t}: a partial slot written != once"
            assert np.all(part_tok[sl] == t)
            assert np.all(part_c[sl].sum(axis=0) == exp_cnt[t]), f"token {t}: key count"
            hs = part_h[sl].sum(axis=0, dtype=np.uint64)
            assert np.all(hs == exp_hash[t, kv]), f"token {t}: key set"
    if collect:
        return {"kinds": kinds, "masked": masked, "pcount": pcount}
    return None
