"""Host-side work plans (pkv_plan_build, include/pkv.h) -- CPU only.

The plan is checked against what it must guarantee whatever its heuristics:
every page of every sequence is attended exactly once, in a range or by one
packed warp; split sequences list their ranges' slots for the merge; CTAs
run in order of the pages their busiest warp streams; the sizes follow the
stated formula.
"""
import numpy as np
import pytest

from paged_kv_decode_04_gb300 import binding as B

SMS = 152


def build(lens, max_blocks=128, sms=SMS):
    return B.Plan(np.asarray(lens, np.int32), max_blocks, num_sms=sms)


def coverage(plan, lens, folds=None):
    """Per sequence: the list of (first page, count) pieces the plan attends.
    folds (a dict): filled with b -> (first slot, count) of the partials a
    segment folds into sequence b's output."""
    pieces = {b: [] for b in range(len(lens))}
    slots = {}
    if folds is None:
        folds = {}
    segs = plan.segments() if plan.num_segs else None
    for it in plan.items():
        kind, slot, p0, n = (int(x) for x in it[:4])
        if kind == 2:                                  # a segment CTA
            first, nseg, pages = slot, p0, n
            assert 1 <= nseg <= 4 and not it[4:].any()
            mine = segs[first:first + nseg]
            assert int(mine[:, 3].sum()) == pages
            for b, L, q0, m, sl, nf, fs, z in (tuple(int(x) for x in sg) for sg in mine):
                assert L == lens[b] and z == 0
                pieces[b].append((q0, m))
                if sl >= 0:
                    assert sl not in slots and nf == 0 and fs == 0
                    slots[sl] = (b, q0)
                elif nf > 0:
                    assert b not in folds
                    folds[b] = (fs, nf)
                else:
                    assert fs == 0
            continue
        assert segs is None
        seqs, ls = it[4:8], it[8:12]
        if kind == 0:
            assert len(set(seqs.tolist())) == 1 and len(set(ls.tolist())) == 1
            b = int(seqs[0])
            assert int(ls[0]) == lens[b]
            pieces[b].append((p0, n))
            if slot >= 0:
                assert slot not in slots
                slots[slot] = (b, p0)
        else:
            assert kind == 1 and slot == -1
            for s, L in zip(seqs.tolist(), ls.tolist()):
                if s >= 0:
                    assert L == lens[s]
                    pieces[s].append((0, -(-L // 16)))
    return pieces, slots


@pytest.mark.parametrize("lens", [
    [2048] * 256,
    [2048],
    [37],
    [0, 0, 0],
    [0, 1, 15, 16, 17, 2047, 2048, 300, 128, 129],
    list(np.random.default_rng(1).integers(0, 2049, 300)),
    list(np.random.default_rng(2).permutation(
        np.concatenate([np.random.default_rng(3).integers(16, 129, 115),
                        np.random.default_rng(4).integers(1536, 2049, 13)]))),
])
def test_every_page_once_and_merges_consistent(lens):
    lens = [int(x) for x in lens]
    plan = build(lens)
    assert plan.magic == B.PLAN_MAGIC and plan.batch == len(lens) and plan.max_blocks == 128
    pieces, slots = coverage(plan, lens)
    for b, L in enumerate(lens):
        p = -(-L // 16)
        got = sorted(pieces[b])
        assert len(got) >= 1, b                    # even an empty sequence gets its zero row
        covered = []
        for p0, n in got:
            covered += list(range(p0, p0 + n))
        assert covered == list(range(p)), (b, got)
    merged = set()
    for b, first, nr, zero in plan.merges().tolist():
        assert zero == 0 and nr >= 2 and b not in merged
        merged.add(b)
        assert [slots[first + r][0] for r in range(nr)] == [b] * nr
        assert [slots[first + r][1] for r in range(nr)] == sorted(p0 for p0, _ in pieces[b])
    split = {b for b in range(len(lens)) if len(pieces[b]) > 1}
    assert split == merged
    assert plan.num_slots == len(slots)
    assert plan.workspace_bytes == plan.num_slots * 32 * 66 * 4
    for it in plan.items():                        # words 12..15 are reserved zeros
        assert not it[12:].any()
    assert plan.num_shared == 0
    assert plan.bytes_used == 4 * (12 + 16 * plan.num_items + 4 * plan.num_merges
                                   + 8 * plan.num_segs)


def expected_sizes(lens, sms, max_blocks=128):
    """The stated rule, written out: the smallest work unit u >= ceil(P / (2 SMs))
    whose plan has at most 4 * SMs CTAs (8 per item), else the widest ranges."""
    pages = [-(-int(L) // 16) for L in lens]
    P = sum(pages)

    def sizes(u):
        R = min(max_blocks, 1024, max(min(8, max_blocks), 4 * u))
        return R, min(16, max(1, R // 4))

    def items(u):
        R, pack = sizes(u)
        n_packed = sum(1 for p in pages if p <= pack)
        return sum(-(-p // R) for p in pages if p > pack) + -(-n_packed // 4)

    u = max(1, -(-P // (2 * sms)))
    umax = max(u, -(-max_blocks // 4))
    while u < umax and items(u) * 8 > 4 * sms:
        u += 1
    return sizes(u)


def test_sizes_follow_the_formula():
    rng = np.random.default_rng(9)
    for _ in range(50):
        n = int(rng.integers(1, 400))
        lens = rng.integers(0, 2049, n)
        sms = int(rng.choice([1, 16, 132, 152]))
        plan = build(lens, sms=sms)
        if plan.num_segs:                          # big layers: a segment plan (tested below)
            continue
        R, pack = expected_sizes(lens, sms)
        assert plan.range_pages == R
        for it in plan.items():
            if it[0] == 0:
                assert 1 <= it[3] <= R
                assert -(-int(it[8]) // 16) > pack    # longer sequences only
            else:
                for L in it[8:12]:
                    assert -(-int(L) // 16) <= pack


def busiest_warp_pages(item):
    if item[0] == 0:
        return -(-int(item[3]) // 4)
    return max(-(-int(L) // 16) for L in item[8:12])


@pytest.mark.parametrize("seed", [5, 6, 7])
def test_order_busiest_warp_first(seed):
    rng = np.random.default_rng(seed)
    # about 1100 pages: below the segment plans' threshold at 152 SMs
    lens = np.concatenate([rng.integers(0, 200, 100), rng.integers(1000, 2049, 5)])
    it = build(rng.permutation(lens)).items()
    assert (it[:, 0] != 2).all()
    work = [busiest_warp_pages(x) for x in it]
    assert work == sorted(work, reverse=True)
    for a, b in zip(it[:-1], it[1:]):              # ranges before packed items on ties
        if busiest_warp_pages(a) == busiest_warp_pages(b):
            assert a[0] <= b[0]


def test_uniform_batch_is_one_segment_per_sequence():
    # 256 x 128 pages on 152 SMs: bins of 128 pages fit one wave of two CTAs
    # per SM, so every sequence is one whole segment and nothing is merged
    plan = build([2048] * 256)
    assert plan.num_segs == 256 and plan.num_items == 256
    assert plan.num_merges == 0 and plan.num_slots == 0
    sg = plan.segments()
    assert sorted(sg[:, 0].tolist()) == list(range(256))
    assert set(sg[:, 3].tolist()) == {128} and set(sg[:, 4].tolist()) == {-1}
    assert set(plan.items()[:, 2].tolist()) == {1}


def test_single_long_sequence_is_split_in_equal_ranges():
    plan = build([2048])
    assert plan.range_pages == 8 and plan.num_items == 16
    assert plan.merges().tolist() == [[0, 0, 16, 0]]
    assert plan.items()[:, 2].tolist() == list(range(0, 128, 8))


def test_same_lengths_same_bytes():
    lens = np.random.default_rng(6).integers(0, 2049, 77)
    assert np.array_equal(build(lens).host, build(lens).host)


def test_invalid_inputs():
    with pytest.raises(B.PkvError):
        build([-1])
    with pytest.raises(B.PkvError):
        build([2049])                               # past the table
    with pytest.raises(B.PkvError):
        build([16], max_blocks=0)
    lib = B.lib()
    assert lib.pkv_plan_bytes(0, 128) == 0
    import ctypes
    lens = np.array([16], np.int32)
    buf = np.zeros(64, np.int32)
    rc = lib.pkv_plan_build(lens.ctypes.data_as(ctypes.c_void_p), 1, 128, SMS,
                            buf.ctypes.data_as(ctypes.c_void_p), 16)   # too small
    assert rc == B.PKV_EINVAL
    assert lib.pkv_plan_workspace_bytes(buf.ctypes.data_as(ctypes.c_void_p)) == \
        ctypes.c_size_t(-1).value                   # no magic


def test_wide_tables_cap_the_range():
    # max_blocks past the kernel's 1024-entry page list: ranges stay <= 1024
    plan = build([65536] * 2, max_blocks=4096, sms=1)
    assert plan.range_pages == 1024
    assert max(int(n) for n in plan.items()[:, 3]) <= 1024


# ------------------------------------------------ host table check (pkv_check_tables) --

def test_check_tables_accepts_a_valid_batch():
    from paged_kv_decode_04_gb300 import synth
    w = synth.make_workload("small", 0)
    B.check_tables(w.block_tables[0], w.seq_lens, w.num_pages)


@pytest.mark.parametrize("case", ["negative_len", "long_len", "negative_page", "page_past_pool"])
def test_check_tables_names_the_first_bad_entry(case):
    lens = np.array([40, 17, 0, 33], np.int32)
    bt = np.full((4, 8), -1, np.int32)
    bt[0, :3] = [5, 6, 7]
    bt[1, :2] = [1, 2]
    bt[3, :3] = [9, 10, 11]
    B.check_tables(bt, lens, 64)                       # entries past a length are never read
    if case == "negative_len":
        lens[2] = -1
        want = "sequence 2: length -1"
    elif case == "long_len":
        lens[1] = 8 * 16 + 1
        want = "sequence 1: length 129"
    elif case == "negative_page":
        bt[3, 2] = -4
        want = "sequence 3, block 2: page -4"
    else:
        bt[1, 1] = 64
        want = "sequence 1, block 1: page 64"
    with pytest.raises(B.PkvError) as e:
        B.check_tables(bt, lens, 64)
    assert want in str(e.value) and e.value.status == B.PKV_EINVAL


def test_plan_built_into_a_caller_buffer_is_the_same_plan():
    lens = np.random.default_rng(31).integers(0, 2049, 90).astype(np.int32)
    nbytes = B.plan_bytes(len(lens), 128)
    raw = np.zeros(nbytes // 4 + 8, np.int32)
    off = (-raw.ctypes.data % 16) // 4
    p = B.Plan(lens, 128, num_sms=SMS, out=raw[off:])
    q = B.Plan(lens, 128, num_sms=SMS)
    assert np.array_equal(p.host, q.host) and p.workspace_bytes == q.workspace_bytes
    assert np.shares_memory(p.host, raw)
    with pytest.raises(ValueError):                 # too small
        B.Plan(lens, 128, num_sms=SMS, out=raw[off:off + 8])
    with pytest.raises(ValueError):                 # misaligned
        B.Plan(lens, 128, num_sms=SMS, out=raw[off + 1:])
    with pytest.raises(ValueError):                 # wrong type
        B.Plan(lens, 128, num_sms=SMS, out=raw[off:].view(np.float32))


# ------------------------------------------- shared prefixes (pkv_plan_build_shared) --

def shared_case(seed, groups, own, mb=128):
    """Consecutive groups of sequences whose tables start with the same pages:
    groups = [(size, shared pages)], own = each sequence's own pages count
    range; returns lens, tables."""
    rng = np.random.default_rng(seed)
    lens, rows, nxt = [], [], 0
    for size, k in groups:
        common = list(range(nxt, nxt + k))
        nxt += k
        for _ in range(size):
            o = int(rng.integers(own[0], own[1] + 1))
            row = common + list(range(nxt, nxt + o))
            nxt += o
            lens.append(16 * (k + o) - int(rng.integers(0, 16)))
            rows.append(row + [-1] * (mb - len(row)))
    return np.asarray(lens, np.int32), np.asarray(rows, np.int32)


def shared_coverage(plan, lens, bt, folds=None):
    pieces, slots = coverage(plan, lens, folds)
    for it in plan.shared().tolist():
        members, p0, n = it[0], it[1], it[2]
        seqs, sl = it[4:4 + members], it[20:20 + members]
        assert 2 <= members <= 16 and all(x == -1 for x in it[4 + members:20])
        assert seqs == list(range(seqs[0], seqs[0] + members))       # consecutive
        for m, (b, slot) in enumerate(zip(seqs, sl)):
            assert np.array_equal(bt[b, p0:p0 + n], bt[seqs[0], p0:p0 + n])
            assert p0 + n <= -(-int(lens[b]) // 16) - 1                # never the last page
            assert slot not in slots
            slots[slot] = (b, p0)
            pieces[b].append((p0, n))
    return pieces, slots


@pytest.mark.parametrize("seed,groups,own", [
    (0, [(16, 96)] * 4, (32, 32)),            # the prefix workload's groups, fewer of them
    (0, [(16, 96)] * 16, (32, 32)),           # the prefix workload: a segment plan
    (4, [(16, 40)] * 12 + [(2, 20)] * 8, (20, 80)),    # segments, some members split
    (1, [(3, 20), (1, 5), (8, 40), (2, 16)], (1, 60)),
    (2, [(5, 1000)], (1, 3)),                 # long prefixes: several shared ranges
])
def test_shared_plan_covers_every_page_once(seed, groups, own):
    mb = 2048 if seed == 2 else 128
    lens, bt = shared_case(seed, groups, own, mb)
    plan = B.Plan(lens, mb, num_sms=SMS, block_tables=bt, min_shared_pages=16)
    assert plan.num_shared > 0
    folds = {}
    pieces, slots = shared_coverage(plan, lens, bt, folds)
    for b, L in enumerate(lens.tolist()):
        covered = []
        for p0, n in sorted(pieces[b]):
            covered += list(range(p0, p0 + n))
        assert covered == list(range(-(-L // 16))), b
    merged = {}
    for b, first, nr, zero in plan.merges().tolist():
        assert zero == 0 and b not in merged
        merged[b] = [slots[first + r] for r in range(nr)]
        assert all(x[0] == b for x in merged[b])
        assert [x[1] for x in merged[b]] == sorted(x[1] for x in merged[b])
    members = {int(x) for it in plan.shared() for x in it[4:4 + it[0]]}
    # every member is merged, or (a segment plan, its own pages one segment)
    # its segment folds exactly its shared ranges' partials, in page order
    assert members <= set(merged) | set(folds) and not set(merged) & set(folds)
    for b, (first, nf) in folds.items():
        assert b in members
        got = [slots[first + r] for r in range(nf)]
        assert all(x[0] == b for x in got)
        assert [x[1] for x in got] == sorted(x[1] for x in got)
        assert len(pieces[b]) == nf + 1
    if plan.num_segs:   # members fold, or (cut into pieces) are merged
        assert len(folds) + len(members & set(merged)) == len(members)
    if groups == [(16, 96)] * 16:
        assert plan.num_merges == 0 and len(folds) == 256
    assert plan.num_slots == len(slots)
    assert plan.bytes_used == 4 * (12 + 16 * plan.num_items + 4 * plan.num_merges
                                   + 36 * plan.num_shared + 8 * plan.num_segs)
    assert plan.shared_pages == max(int(n) for n in plan.shared()[:, 2])


def test_shared_groups_follow_the_rule():
    lens, bt = shared_case(3, [(20, 30), (2, 10), (3, 17)], (2, 5))
    plan = B.Plan(lens, 128, num_sms=SMS, block_tables=bt, min_shared_pages=16)
    sh = plan.shared()
    firsts = sorted({(int(it[4]), int(it[0])) for it in sh})
    # 20 sharing 30 pages: groups of 16 and 4; 2 sharing 10 < 16 pages: none;
    # 3 sharing 17: one group
    assert firsts == [(0, 16), (16, 4), (22, 3)]
    ends = sorted(int(it[1]) + int(it[2]) for it in sh if it[4] == 22)
    assert ends[-1] == 17 and int(min(it[1] for it in sh if it[4] == 22)) == 0


def test_without_tables_or_sharing_the_plan_is_the_plain_one():
    lens = np.random.default_rng(4).integers(1, 2049, 60).astype(np.int32)
    bt = np.arange(60 * 128, dtype=np.int32).reshape(60, 128)     # nothing shared
    a = B.Plan(lens, 128, num_sms=SMS)
    b = B.Plan(lens, 128, num_sms=SMS, block_tables=bt)
    assert a.num_shared == b.num_shared == 0
    assert np.array_equal(a.host, b.host)


@pytest.mark.parametrize("sms", [1, 100, 132, 152])
def test_shared_ranges_fill_one_wave(sms):
    # the prefix workload: 16 groups of 16 sequences sharing 96 pages, 128
    # (group, kv head) pairs.  With at least 128 SMs the shared-prefix CTAs
    # fit one per SM and the plan runs its segment CTAs beside them, one per
    # SM too (layout 1); otherwise the shared-prefix CTAs run first, two per
    # SM (layout 0).  Each group's prefix is cut into as many near-equal
    # ranges as keep its CTAs within that one wave: one range of 96 pages here.
    from paged_kv_decode_04_gb300 import synth
    w = synth.make_workload("prefix", 0)
    plan = B.Plan(w.seq_lens, w.max_blocks, num_sms=sms, block_tables=w.block_tables[0])
    sh = plan.shared()
    beside = sms >= 128
    assert plan.layout == (1 if beside else 0)
    assert plan.num_shared == 16
    assert all(int(it[0]) == 16 for it in sh)
    assert sorted({int(it[2]) for it in sh}) == [96]
    assert plan.num_segs > 0
    if beside:
        assert plan.num_shared * 8 <= sms and plan.num_items <= sms
    elif sms > 1:
        assert plan.num_shared * 8 <= 2 * sms or plan.num_shared == 16
    for g in range(16):   # each group's ranges tile its 96 shared pages
        mine = sorted((int(it[1]), int(it[2])) for it in sh if int(it[4]) == 16 * g)
        assert mine[0][0] == 0 and all(a + n == b for (a, n), (b, _) in zip(mine, mine[1:]))
        assert mine[-1][0] + mine[-1][1] == 96


@pytest.mark.parametrize("groups, sms, layout, ranges", [
    (8, 152, 1, 2),      # 64 pairs: beside, two ranges of 48 per group (128 CTAs)
    (8, 64, 1, 1),       # 64 pairs on 64 SMs: beside, one range each
    (32, 152, 0, 1),     # 256 pairs > 152 SMs: shared-prefix CTAs first
    (4, 152, 1, 4),      # 2048 own pages, under the 16-pages-per-SM gate of other segment
                         # plans: beside all the same (bins of 16, members cut in two)
])
def test_beside_layout_when_the_shared_ctas_fit_one_per_sm(groups, sms, layout, ranges):
    lens, bt = shared_case(5, [(16, 96)] * groups, (32, 32))
    plan = B.Plan(lens, 128, num_sms=sms, block_tables=bt, min_shared_pages=16)
    assert plan.num_segs > 0 and plan.num_shared == groups * ranges
    assert plan.layout == layout
    if groups == 4:
        assert plan.range_pages == 16 and plan.num_merges == 64
    if layout == 1:
        assert plan.num_shared * 8 <= sms and plan.num_items <= sms
    pieces, slots = shared_coverage(plan, lens, bt)


def _kernels_for(plan_words, batch, mb=128):
    """pkv_attention_kernels on a copy of the plan words (host code only):
    None when the library refuses the plan."""
    import ctypes
    raw = np.zeros(plan_words.shape[0] + 4, dtype=np.int32)
    off = (-raw.ctypes.data % 16) // 4
    buf = raw[off:off + plan_words.shape[0]]
    buf[:] = plan_words
    return B.lib().pkv_attention_kernels(batch, mb, 0, buf.ctypes.data_as(ctypes.c_void_p))


def test_damaged_plans_are_refused_before_any_launch():
    # a plan is plain data: every index a kernel would take from it (sequence,
    # page range, partial slot, member count) and the byte count its header
    # states are checked on the host, so a hand-made or damaged plan is
    # refused instead of sending a kernel outside its buffers
    lens, bt = shared_case(0, [(16, 96)] * 2, (32, 32))
    lens = np.concatenate([lens, np.array([2048, 40, 3], np.int32)])
    extra = np.arange(3 * 128, dtype=np.int32).reshape(3, 128) + 100000
    bt = np.concatenate([bt, extra])
    plan = B.Plan(lens, 128, num_sms=SMS, block_tables=bt, min_shared_pages=16)
    batch = len(lens)
    assert plan.num_shared > 0 and plan.num_merges > 0
    kinds = plan.items()[:, 0]
    assert (kinds == 0).any() and (kinds == 1).any()
    good = plan.host.copy()
    assert _kernels_for(good, batch) is not None
    it0 = B.PLAN_HEADER_WORDS
    rng_i = it0 + 16 * int(np.flatnonzero(kinds == 0)[0])
    pk_i = it0 + 16 * int(np.flatnonzero(kinds == 1)[0])
    mg = it0 + 16 * plan.num_items
    sh = mg + 4 * plan.num_merges
    damage = {
        "bytes_used": (7, int(good[7]) - 4),
        "range item sequence": (rng_i + 4, batch),
        "range item negative sequence": (rng_i + 4, -1),
        "range longer than the page list": (rng_i + 3, plan.range_pages + 1),
        "range past the table": (rng_i + 2, 128),
        "range item slot": (rng_i + 1, plan.num_slots),
        "unknown item kind": (rng_i, 2),
        "packed item sequence": (pk_i + 4, batch + 7),
        "packed item length": (pk_i + 8, 128 * 16 + 1),
        "merge sequence": (mg, batch),
        "merge slots": (mg + 2, plan.num_slots + 1),
        "shared members": (sh, 17),
        "no shared members": (sh, 0),
        "shared range": (sh + 2, plan.shared_pages + 1),
        "shared member sequence": (sh + 5, batch),
        "shared member slot": (sh + 21, plan.num_slots),
        "merges beyond the batch": (4, batch + 1),
    }
    for what, (idx, value) in damage.items():
        bad = good.copy()
        bad[idx] = value
        assert _kernels_for(bad, batch) is None, what


def test_rebuild_in_place_gives_the_plan_of_the_new_lengths():
    # a serving loop rebuilds the step's plan into the same (pinned) buffer
    rng = np.random.default_rng(9)
    a = rng.integers(1, 2049, 100).astype(np.int32)
    b = rng.integers(1, 2049, 100).astype(np.int32)
    p = B.Plan(a, 128, num_sms=SMS)
    buf = p.host.base if p.host.base is not None else p.host
    p.rebuild(b)
    q = B.Plan(b, 128, num_sms=SMS)
    assert np.array_equal(p.host, q.host)
    assert (p.num_items, p.num_merges, p.workspace_bytes) == (q.num_items, q.num_merges,
                                                              q.workspace_bytes)
    assert np.shares_memory(p.host, buf)
    # with shared prefixes: the tables' groups are found again
    lens, bt = shared_case(1, [(3, 20), (1, 5), (8, 40), (2, 16)], (1, 60))
    p = B.Plan(lens, 128, num_sms=SMS, block_tables=bt)
    lens2 = lens.copy()
    lens2[-1] += 1
    p.rebuild(np.ascontiguousarray(lens2), np.ascontiguousarray(bt))
    q = B.Plan(lens2, 128, num_sms=SMS, block_tables=bt)
    assert np.array_equal(p.host, q.host) and p.num_shared == q.num_shared > 0


# ---------------------------------------------------------- segment plans --

@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_segment_plans_pack_one_wave_of_near_equal_ctas(seed):
    # large ragged layers get segment plans: every page once, at most 4
    # segments and range_pages pages per CTA, CTAs largest first, at most two
    # CTAs per SM whenever the bins can be that small, split sequences merged
    rng = np.random.default_rng(seed)
    lens = rng.integers(200, 2049, int(rng.integers(100, 300))).astype(np.int32)
    lens[:5] = 0                                   # empty sequences get a segment too
    plan = build(lens)
    assert plan.num_segs > 0
    pieces, slots = coverage(plan, [int(x) for x in lens])
    for b, L in enumerate(lens.tolist()):
        covered = sorted(p for p0, n in pieces[b] for p in range(p0, p0 + n))
        assert covered == list(range(-(-L // 16)))
    it = plan.items()
    pages = it[:, 3]
    assert pages.max() == plan.range_pages and list(pages) == sorted(pages, reverse=True)
    assert (it[:, 2] <= 4).all()
    P = int(sum(-(-int(L) // 16) for L in lens))
    if plan.range_pages < 1024 and plan.range_pages < max(-(-int(L) // 16) for L in lens):
        assert plan.num_items <= 2 * SMS
    merged = {int(m[0]): int(m[2]) for m in plan.merges()}
    for b in range(len(lens)):
        if len(pieces[b]) > 1:
            assert merged[b] == len(pieces[b])
        else:
            assert b not in merged
    assert plan.num_slots == sum(merged.values())
    assert P == int(pages.sum())


def test_plan_kind_follows_the_bin_size():
    # a segment plan only where its bins hold at least 16 pages: the mixed
    # batch (2067 pages over 152 SMs) keeps the per-(item, kv head) plan;
    # 256 x 128 pages is one whole sequence per segment CTA, nothing merged;
    # 1024 x 16 pages packs about three sequences per CTA into one wave
    from paged_kv_decode_04_gb300 import synth
    w = synth.make_workload("mix", 0)
    mix = B.Plan(w.seq_lens, w.max_blocks, num_sms=SMS)
    assert mix.num_segs == 0 and set(mix.items()[:, 0].tolist()) == {0, 1}
    peak = build([2048] * 256)
    assert peak.num_segs == peak.num_items == 256 and peak.num_merges == 0
    many = build([256] * 1024)
    assert many.num_segs == 1024 and many.num_items <= 2 * SMS and many.num_merges == 0
    assert many.range_pages >= 16 and many.items()[:, 2].max() <= 4


def test_damaged_segment_plans_are_refused():
    lens = np.random.default_rng(12).integers(200, 2049, 150).astype(np.int32)
    plan = build(lens)
    batch = len(lens)
    good = plan.host.copy()
    assert _kernels_for(good, batch) == "paged_decode_segments_kernel+merge_plan_kernel".encode()
    sg0 = B.PLAN_HEADER_WORDS + 16 * plan.num_items + 4 * plan.num_merges
    split = int(np.flatnonzero(plan.segments()[:, 4] >= 0)[0])
    damage = {
        "item kind": (12, 0),
        "no segments": (14, 0),
        "five segments": (14, 5),
        "item pages": (15, int(good[15]) + 1),
        "segments past the section": (13, plan.num_segs),
        "segment sequence": (sg0, batch),
        "segment length": (sg0 + 1, 2049),
        "segment past its sequence": (sg0 + 2, 128),
        "segment slot": (sg0 + 8 * split + 4, plan.num_slots),
        "segment count in the header": (10, plan.num_segs + 1),
    }
    for what, (idx, value) in damage.items():
        bad = good.copy()
        bad[idx] = value
        assert _kernels_for(bad, batch) is None, what


def test_damaged_fold_words_are_refused():
    # a segment that folds partials into its output names slots inside the
    # plan's partial area and writes the output itself (slot -1); reserved
    # words stay zero
    lens, bt = shared_case(0, [(16, 96)] * 16, (32, 32))
    plan = B.Plan(lens, 128, num_sms=SMS, block_tables=bt, min_shared_pages=16)
    batch = len(lens)
    good = plan.host.copy()
    assert _kernels_for(good, batch) == \
        "paged_decode_shared_kernel+paged_decode_segments_kernel".encode()
    sg0 = (B.PLAN_HEADER_WORDS + 16 * plan.num_items + 4 * plan.num_merges
           + 36 * plan.num_shared)
    segs = plan.segments()
    f = int(np.flatnonzero((segs[:, 5] > 0) & (segs[:, 6] > 0))[0])
    at = sg0 + 8 * f
    damage = {
        "fold past the slots": (at + 6, plan.num_slots - int(segs[f, 5]) + 1),
        "negative fold slot": (at + 6, -1),
        "negative fold count": (at + 5, -1),
        "fold with a partial of its own": (at + 4, 0),
        "reserved word": (at + 7, 1),
    }
    for what, (idx, value) in damage.items():
        bad = good.copy()
        bad[idx] = value
        assert _kernels_for(bad, batch) is None, what
    unfolded = good.copy()
    unfolded[at + 5] = 0
    assert _kernels_for(unfolded, batch) is None      # fold slot left without a fold
    unfolded[at + 6] = 0
    assert _kernels_for(unfolded, batch) is not None


def test_concurrent_builds_match_sequential_ones():
    """The planner keeps reusable buffers per calling thread: plans built
    from many threads at once (ctypes drops the GIL for the call) are the
    plans built one at a time."""
    import threading
    rng = np.random.default_rng(11)
    cases = [(np.full(256, 2048, np.int32), None),                       # segment plan
             (rng.integers(1, 2049, 1024).astype(np.int32), None),       # packed bins
             (np.concatenate([rng.integers(16, 129, 115),
                              rng.integers(1536, 2049, 13)]).astype(np.int32), None),
             (np.full(64, 2048, np.int32), None),                        # split sequences
             shared_case(3, [(16, 96)] * 16, (32, 32)),
             shared_case(4, [(5, 20), (1, 0), (9, 40), (3, 17)], (1, 80))]

    def plan_bytes(lens, bt):
        p = B.Plan(lens, 128, num_sms=SMS, block_tables=bt)
        return p.host.tobytes()

    want = [plan_bytes(lens, bt) for lens, bt in cases]
    bad = []

    def worker(t):
        order = np.random.default_rng(t).permutation(len(cases))
        for _ in range(20):
            for i in order:
                if plan_bytes(*cases[i]) != want[i]:
                    bad.append((t, int(i)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(8)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not bad


def test_layout_word_is_checked():
    # header word 11: 0 (shared-prefix CTAs first) or 1 (segment CTAs beside
    # them), and 1 only for a shared-prefix plan of segment CTAs
    lens, bt = shared_case(0, [(16, 96)] * 16, (32, 32))
    beside = B.Plan(lens, 128, num_sms=SMS, block_tables=bt, min_shared_pages=16)
    assert beside.layout == 1
    good = beside.host.copy()
    assert _kernels_for(good, len(lens)) is not None
    seq = good.copy()
    seq[11] = 0                      # the same plan run in sequence is still a plan
    assert _kernels_for(seq, len(lens)) is not None
    for bad_layout in (2, -1):
        bad = good.copy()
        bad[11] = bad_layout
        assert _kernels_for(bad, len(lens)) is None
    plain = B.Plan(np.full(256, 2048, np.int32), 128, num_sms=SMS)      # segments, no groups
    assert plain.num_segs > 0 and plain.num_shared == 0 and plain.layout == 0
    bad = plain.host.copy()
    bad[11] = 1                      # nothing to run beside
    assert _kernels_for(bad, 256) is None
    # per-head items beside the shared-prefix CTAs: either layout is a valid plan
    small_lens, small_bt = shared_case(1, [(3, 20), (1, 5), (8, 40), (2, 16)], (1, 60))
    small = B.Plan(small_lens, 128, num_sms=SMS, block_tables=small_bt, min_shared_pages=16)
    assert small.num_shared > 0 and small.num_segs == 0 and small.layout == 1
    seq = small.host.copy()
    seq[11] = 0
    assert _kernels_for(seq, len(small_lens)) == \
        b"paged_decode_shared_kernel+paged_decode_kernel+merge_plan_kernel"
    bad = small.host.copy()
    bad[11] = 2
    assert _kernels_for(bad, len(small_lens)) is None


@pytest.mark.parametrize("groups", [1, 2])
def test_small_shared_batches_run_per_head_items_beside(groups):
    # 16 or 32 sequences (512 or 1024 own pages): bins of one CTA per SM would
    # hold fewer than 16 pages, so no segment plan; the per-(item, kv head)
    # CTAs (two per SM next to a shared-prefix CTA) run beside the
    # shared-prefix CTAs (layout 1), and the merge after them
    lens, bt = shared_case(5, [(16, 96)] * groups, (32, 32))
    plan = B.Plan(lens, 128, num_sms=SMS, block_tables=bt, min_shared_pages=16)
    assert plan.num_segs == 0 and plan.layout == 1 and plan.num_merges == 16 * groups
    assert plan.num_shared * 8 <= SMS
    assert plan.num_items * 8 <= 4 * SMS - 2 * plan.num_shared * 8
    shared_coverage(plan, lens, bt)


@pytest.mark.parametrize("seed", range(40))
def test_random_shared_plans_keep_their_layout_rules(seed):
    # random groups (2..16 members, 16..100 shared pages), singletons, own
    # tails of 1..80 pages, planned for a random SM count: every page is
    # attended once; a beside plan (layout 1) has at most one shared-prefix
    # CTA per SM, and one segment CTA per SM if it has segments; segment bins
    # hold at least 16 pages;
    # members either fold or are merged; the library accepts the plan
    rng = np.random.default_rng(500 + seed)
    sms = int(rng.choice([8, 16, 32, 64, 100, 132, 152]))
    groups = []
    for _ in range(int(rng.integers(1, 9))):
        if rng.random() < 0.3:
            groups.append((1, 0))
        groups.append((int(rng.integers(2, 17)), int(rng.integers(16, 101))))
    kmax = max(k for _, k in groups)
    own = (1, int(min(rng.choice([8, 30, 80]), 127 - kmax)))   # within the 128-entry table
    lens, bt = shared_case(int(rng.integers(0, 1 << 30)), groups, own)
    plan = B.Plan(lens, 128, num_sms=sms, block_tables=bt, min_shared_pages=16)
    folds = {}
    pieces, slots = shared_coverage(plan, lens, bt, folds)
    for b, L in enumerate(lens.tolist()):
        covered = sorted(p for p0, n in pieces[b] for p in range(p0, p0 + n))
        assert covered == list(range(-(-L // 16))), b
    members = {int(x) for it in plan.shared() for x in it[4:4 + it[0]]}
    merged = {int(m[0]) for m in plan.merges()}
    assert members <= merged | set(folds) and not merged & set(folds)
    if plan.layout == 1:
        assert plan.num_shared > 0 and plan.num_shared * 8 <= sms
        if plan.num_segs:
            assert plan.num_items <= sms and plan.range_pages >= 16
    elif plan.num_segs:   # one wave of two per SM when some bin size fits it
        assert plan.range_pages >= 16
    assert _kernels_for(plan.host.copy(), len(lens)) is not None
