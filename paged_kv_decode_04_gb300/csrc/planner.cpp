// planner.cpp -- host-side work plans for ragged decode batches (the
// pkv_plan_* entry points of include/pkv.h).  Plain C++17, no CUDA.
//
// The attention kernel handles one (work item, kv head) per CTA.  A work
// item is either a range of logical pages of one sequence, shared by the
// CTA's 4 warps, or up to 4 short sequences, one per warp.  The plan below
// is made from the lengths the caller already holds on the host (its
// scheduler allocated every page), so the grid holds exactly the needed
// CTAs and the longest work starts first.
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "pkv.h"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kMinRangePages = 8;     // shortest range worth a CTA of its own
constexpr int kResidentPerSm = 4;     // attention CTAs resident per SM (shallow ring)
constexpr int kMaxRangePages = 1024;  // the kernel's shared page list
constexpr int kMinSegPages = 4;       // smallest bin size tried for a segment plan
constexpr int kMinSegBinPages = 16;   // smallest bin size a segment plan is used with
constexpr int kPerHeadBesideCtasPerSm = 2;  // per-head CTAs next to a shared-prefix CTA (registers)

struct Range {
  int b, L, p_begin, n, slot;
};

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// Stable counting sort of v by key(x) in [0, nkeys), ascending; the keys here
// are small page counts, so this is a few linear passes (a comparison sort of
// a 256-sequence batch took most of the plan's host time).  Its buffers are
// the calling thread's and keep their capacity from one plan to the next.
template <typename T, typename Key>
void counting_sort(std::vector<T>& v, int nkeys, Key key) {
  static thread_local std::vector<int> first_buf;
  static thread_local std::vector<T> out_buf;
  std::vector<int>& first = first_buf;  // thread-local lookups once, not per element
  std::vector<T>& out = out_buf;
  first.assign(static_cast<size_t>(nkeys) + 1, 0);
  for (const T& x : v) ++first[static_cast<size_t>(key(x)) + 1];
  for (int k = 0; k < nkeys; ++k) first[k + 1] += first[k];
  out.resize(v.size());
  for (const T& x : v) out[first[key(x)]++] = x;
  std::copy(out.begin(), out.end(), v.begin());
}

}  // namespace

size_t plan_bytes(int batch, int max_blocks) {
  if (batch < 1 || max_blocks < 1) return 0;
  const int rmin = max_blocks < kMinRangePages ? max_blocks : kMinRangePages;
  // range / packed items, or segment CTAs (at most one per segment)
  const size_t pieces = static_cast<size_t>(batch) * (ceil_div(max_blocks, rmin) + 1);
  const size_t items = pieces + 1;
  // shared-prefix items: at most one per (group of two or more, range)
  const size_t shared = static_cast<size_t>(batch / 2) * ceil_div(max_blocks, rmin);
  return 4 * (kPlanHeaderWords + items * kPlanItemWords +
              static_cast<size_t>(batch) * kPlanMergeWords + shared * kPlanSharedWords +
              pieces * kPlanSegWords);
}

// Sizes for work unit u (the pages one warp streams): ranges of R = 4 u
// pages (at least kMinRangePages, at most the table width and
// kMaxRangePages), sequences of at most R / 4 pages (and kPackPages) packed
// one per warp.
struct Sizes {
  int range, pack_max;
};

Sizes sizes_for(long long u, int max_blocks) {
  const int rmin = max_blocks < kMinRangePages ? max_blocks : kMinRangePages;
  const int rmax = max_blocks < kMaxRangePages ? max_blocks : kMaxRangePages;
  long long R = u * kPlanWarps;
  R = std::max<long long>(R, rmin);
  R = std::min<long long>(R, rmax);
  const int range = static_cast<int>(R);
  return {range, std::min(kPackPages, std::max(1, range / kPlanWarps))};
}

// Work items (CTAs per kv head) of the plan for sizes z.
long long count_items(const std::vector<int>& pages, Sizes z) {
  long long items = 0, packed = 0;
  for (int p : pages) {
    if (p <= z.pack_max) ++packed;
    else items += (p + z.range - 1) / z.range;
  }
  return items + (packed + kPlanWarps - 1) / kPlanWarps;
}

// A run of consecutive sequences whose block tables start with the same k
// pages (k at least the minimum asked for, and below every member's last
// page, which takes the step's append and so stays its own).
struct SharedGroup {
  int first, members, k;
};

// Shared-prefix items at `item`: {members, p_begin, n, 0, seq[16], slot[16]},
// range r of group gi taking slot slot_base[member] + r; returns the end.
int32_t* write_shared_items(const std::vector<SharedGroup>& groups,
                            const std::vector<int>& shared_ranges,
                            const std::vector<int>& slot_base, int32_t* item) {
  for (size_t gi = 0; gi < groups.size(); ++gi) {
    const SharedGroup& g = groups[gi];
    const int ns = shared_ranges[gi];
    const int base = g.k / ns, extra = g.k % ns;
    int begin = 0;
    for (int r = 0; r < ns; ++r) {
      const int n = base + (r < extra ? 1 : 0);
      item[0] = g.members;
      item[1] = begin;
      item[2] = n;
      for (int m = 0; m < kSharedMembers; ++m) {
        const bool has = m < g.members;
        item[4 + m] = has ? g.first + m : -1;
        item[4 + kSharedMembers + m] = has ? slot_base[g.first + m] + r : -1;
      }
      begin += n;
      item += kPlanSharedWords;
    }
  }
  return item;
}

// A piece of a sequence's own pages for the segment kernel.
struct Piece {
  int b, p_begin, n;
};

// The pieces for bins of T pages: each sequence's own pages [start, start +
// own) whole, or cut into ceil(own / T) near-equal chunks when longer than T
// (an empty sequence is one piece of no pages, which writes its zero rows),
// largest first (stable), into `pieces`.
void make_pieces(const std::vector<int>& own, const std::vector<int>& start, int T,
                 std::vector<Piece>& pieces) {
  pieces.clear();
  for (size_t b = 0; b < own.size(); ++b) {
    const int p = own[b];
    if (p <= T) {  // whole: no divisions (this runs several times per plan)
      pieces.push_back({static_cast<int>(b), start[b], p});
      continue;
    }
    const int nr = (p + T - 1) / T;
    const int base = p / nr, extra = p % nr;
    int begin = start[b];
    for (int r = 0; r < nr; ++r) {
      const int n = base + (r < extra ? 1 : 0);
      pieces.push_back({static_cast<int>(b), begin, n});
      begin += n;
    }
  }
  counting_sort(pieces, T + 1, [&](const Piece& x) { return T - x.n; });
}

// Best-fit packing of pieces (largest first) into bins of at most T pages and
// kSegMax segments: a piece goes to the open bin with the least room that
// takes it, else to a new bin.  Returns the number of bins; with `bin_of`,
// also each piece's bin.
long long pack_bins(const std::vector<Piece>& pieces, int T, std::vector<int>* bin_of) {
  // the open bins with r pages of room, a stack per r: head[r] the last bin
  // put there, below[bin] the one under it (-1: none); all of it the calling
  // thread's, reused from one packing to the next (the bin-size search packs
  // several times per plan)
  static thread_local std::vector<int> head_buf, below_buf, room_buf, segs_buf;
  static thread_local std::vector<uint64_t> nonempty_buf;
  std::vector<int>& head = head_buf;  // thread-local lookups once, not per piece
  std::vector<int>& below = below_buf;
  std::vector<int>& room = room_buf;
  std::vector<int>& segs = segs_buf;
  std::vector<uint64_t>& nonempty = nonempty_buf;  // bit r: head[r] >= 0
  head.assign(static_cast<size_t>(T) + 1, -1);
  nonempty.assign((static_cast<size_t>(T) >> 6) + 1, 0);
  below.clear();
  room.clear();
  segs.clear();
  auto first_room = [&](int n) {  // the least room >= n held by an open bin, or -1
    for (int w = n >> 6; w < static_cast<int>(nonempty.size()); ++w) {
      uint64_t bits = nonempty[w];
      if (w == (n >> 6)) bits &= ~0ull << (n & 63);
      if (bits) return (w << 6) + __builtin_ctzll(bits);
    }
    return -1;
  };
  if (bin_of != nullptr) bin_of->assign(pieces.size(), -1);
  for (size_t i = 0; i < pieces.size(); ++i) {
    const int n = pieces[i].n;
    int pick = -1;
    const int r = first_room(n);
    if (r >= 0 && r <= T) {
      pick = head[r];
      head[r] = below[pick];
      if (head[r] < 0) nonempty[r >> 6] &= ~(1ull << (r & 63));
    }
    if (pick < 0) {
      pick = static_cast<int>(room.size());
      room.push_back(T);
      segs.push_back(0);
      below.push_back(-1);
    }
    room[pick] -= n;
    segs[pick] += 1;
    if (bin_of != nullptr) (*bin_of)[i] = pick;
    if (segs[pick] < kSegMax) {
      const int rr = room[pick];
      below[pick] = head[rr];
      head[rr] = pick;
      nonempty[rr >> 6] |= 1ull << (rr & 63);
    }
  }
  return static_cast<long long>(room.size());
}

// A packing of the pieces for bins of T pages (T = -1: none yet).
struct Packing {
  int T = -1;
  long long bins = 0;
  std::vector<Piece> pieces;
  std::vector<int> bin_of;
};

// The bin size of a segment plan: the smallest T from max(kMinSegPages,
// ceil(P / C)) up (P: the pages to attend, C = ctas_per_sm CTAs per SM)
// whose bins fit in one wave of C CTAs, else the largest (up to kSegMax x the
// longest sequence, or kSegMaxPages; *fitted says which).  A T whose pieces cannot fit is ruled
// out without packing, by lower bounds on the bins: more than C * T pages;
// or, for k < kSegMax, more than k * C pieces longer than T / (k + 1) (at
// most k of them share a bin); or more than kSegMax * C pieces.  One that
// has at most C pieces fits without packing (best fit opens a bin only for
// a piece that no open bin takes).
int segment_bin_size(const std::vector<int>& own, const std::vector<int>& start, int num_sms,
                     int ctas_per_sm, long long total, Packing& best, bool* fitted = nullptr) {
  const long long C = static_cast<long long>(ctas_per_sm) * num_sms;
  const int max_own = *std::max_element(own.begin(), own.end());
  const int t0 = static_cast<int>(std::min<long long>(
      kSegMaxPages, std::max<long long>(kMinSegPages, (total + C - 1) / C)));
  // past kSegMax x the longest sequence a bin is bounded by its segment count
  const int t1 = std::max(t0, std::min(kSegMax * std::max(max_own, 1), kSegMaxPages));
  // from T = max_own up every sequence is one piece, in the same order
  static thread_local std::vector<Piece> whole_buf;
  static thread_local Packing probe_buf;
  std::vector<Piece>& whole_pieces = whole_buf;
  Packing& probe = probe_buf;
  bool have_whole = false;
  best.T = -1;
  // the sequences by page count: the bounds below take each count once
  static thread_local std::vector<int> seqs_with_buf, counts_buf;
  std::vector<int>& seqs_with = seqs_with_buf;
  std::vector<int>& counts = counts_buf;
  seqs_with.assign(static_cast<size_t>(max_own) + 1, 0);
  counts.clear();
  for (int p : own)
    if (seqs_with[p]++ == 0) counts.push_back(p);
  auto fits = [&](int T) {
    long long cnt[kSegMax + 1] = {};  // k < kSegMax: pieces with (k + 1) n > T; kSegMax: all
    for (int p : counts) {
      const long long m = seqs_with[p];
      const int nr = p > T ? (p + T - 1) / T : 1;
      const int base = nr == 1 ? p : p / nr, extra = nr == 1 ? 0 : p % nr;
      for (int k = 1; k < kSegMax; ++k)
        cnt[k] += m * ((k + 1) * base > T ? nr : ((k + 1) * (base + 1) > T ? extra : 0));
      cnt[kSegMax] += m * nr;
    }
    for (int k = 1; k <= kSegMax; ++k)
      if (cnt[k] > k * C) return false;
    if ((total + T - 1) / T > C) return false;
    if (cnt[kSegMax] <= C) {  // a bin per piece fits: no need to pack
      best.T = -1;            // (the plan packs its own T)
      return true;
    }
    if (T >= max_own) {
      if (!have_whole) {
        make_pieces(own, start, T, whole_pieces);
        have_whole = true;
      }
      probe.pieces = whole_pieces;
    } else {
      make_pieces(own, start, T, probe.pieces);
    }
    probe.T = T;
    probe.bins = pack_bins(probe.pieces, T, &probe.bin_of);
    if (probe.bins > C) return false;
    // the fitting T only decreases as the search goes on: the last one kept
    // is the answer's, which the plan then reuses
    std::swap(best, probe);
    return true;
  };
  // the smallest fitting T, searched first up to the longest sequence (where
  // whole sequences become single pieces), then beyond it
  auto smallest = [&](int lo, int hi) {  // the smallest T in [lo, hi] that fits, or -1
    if (lo > hi || !fits(hi)) return -1;
    while (lo < hi) {
      const int mid = lo + (hi - lo) / 2;
      if (fits(mid)) hi = mid;
      else lo = mid + 1;
    }
    return lo;
  };
  const int whole = std::min(std::max(t0, max_own), t1);
  int T = smallest(t0, whole);
  if (T < 0) T = smallest(whole + 1, t1);
  if (fitted != nullptr) *fitted = T >= 0;
  return T < 0 ? t1 : T;
}

// The segment plan for bins of T pages; bins run largest first.  A sequence
// in more than one piece writes partials to consecutive slots (a group
// member's shared ranges first) and gets a merge entry.  A group member whose
// own pages are one piece folds its shared ranges' partials into its own rows
// and writes its output (the shared-prefix kernel has ended when the segment
// kernel passes its grid wait): its slots hold only those partials, and it
// gets no merge entry.  Any other sequence's segment writes its output.
int build_segments(const int32_t* lens, int batch, int max_blocks, int T,
                   const std::vector<int>& own, const std::vector<int>& start,
                   const std::vector<int>& group_of, const std::vector<SharedGroup>& groups,
                   const std::vector<int>& shared_ranges, int shared_max, int layout,
                   Packing& packing, int32_t* out, size_t out_bytes) {
  if (packing.T != T) {  // not the bin-size search's packing
    make_pieces(own, start, T, packing.pieces);
    packing.T = T;
    packing.bins = pack_bins(packing.pieces, T, &packing.bin_of);
  }
  const std::vector<Piece>& pieces = packing.pieces;
  const std::vector<int>& bin_of = packing.bin_of;
  const int nbins = static_cast<int>(packing.bins);
  // each bin's pieces, in the order they were placed (largest first)
  std::vector<int> by_bin(pieces.size());
  for (size_t i = 0; i < pieces.size(); ++i) by_bin[i] = static_cast<int>(i);
  counting_sort(by_bin, nbins, [&](int i) { return bin_of[i]; });
  std::vector<int> bin_first(static_cast<size_t>(nbins) + 1, 0);
  for (int i : by_bin) ++bin_first[bin_of[i] + 1];
  for (int k = 0; k < nbins; ++k) bin_first[k + 1] += bin_first[k];

  // partial slots: split sequences and group members, in sequence order
  std::vector<int> npieces(batch, 0), slot_base(batch, -1), next_piece(batch, 0);
  for (const Piece& pc : pieces) ++npieces[pc.b];
  std::vector<int32_t> merges;
  int slots = 0;
  for (int b = 0; b < batch; ++b) {
    const int ns = group_of[b] >= 0 ? shared_ranges[group_of[b]] : 0;
    if (npieces[b] > 1) {
      merges.insert(merges.end(), {b, slots, ns + npieces[b], 0});
      slot_base[b] = slots;
      slots += ns + npieces[b];
    } else if (ns > 0) {  // folded by its one own segment
      slot_base[b] = slots;
      slots += ns;
    }
  }
  // a split sequence's pieces take its slots in the order of their pages
  std::vector<int> piece_slot(pieces.size(), -1);
  if (pieces.size() > static_cast<size_t>(batch)) {  // some sequence is split
    std::vector<int> by_page(pieces.size());
    for (size_t i = 0; i < pieces.size(); ++i) by_page[i] = static_cast<int>(i);
    counting_sort(by_page, max_blocks + 1, [&](int i) { return pieces[i].p_begin; });
    for (int i : by_page) {
      const Piece& pc = pieces[i];
      if (npieces[pc.b] < 2) continue;
      const int ns = group_of[pc.b] >= 0 ? shared_ranges[group_of[pc.b]] : 0;
      piece_slot[i] = slot_base[pc.b] + ns + next_piece[pc.b]++;
    }
  }
  // bins largest first (stable)
  std::vector<int> bin_pages(nbins, 0), order(nbins);
  int most = 0;
  for (int k = 0; k < nbins; ++k) {
    for (int j = bin_first[k]; j < bin_first[k + 1]; ++j) bin_pages[k] += pieces[by_bin[j]].n;
    most = std::max(most, bin_pages[k]);
    order[k] = k;
  }
  counting_sort(order, most + 1, [&](int k) { return most - bin_pages[k]; });

  const size_t num_items = static_cast<size_t>(nbins);
  const size_t num_merges = merges.size() / kPlanMergeWords;
  size_t num_shared = 0;
  for (int ns : shared_ranges) num_shared += static_cast<size_t>(ns);
  if (num_items > 65535 || num_shared > 65535) return PKV_EUNSUPPORTED;  // grid limits
  const size_t words = kPlanHeaderWords + num_items * kPlanItemWords + merges.size() +
                       num_shared * kPlanSharedWords + pieces.size() * kPlanSegWords;
  if (words * 4 > out_bytes) return PKV_EINVAL;
  memset(out, 0, words * 4);
  out[0] = static_cast<int32_t>(PKV_PLAN_MAGIC);
  out[1] = batch;
  out[2] = max_blocks;
  out[3] = static_cast<int32_t>(num_items);
  out[4] = static_cast<int32_t>(num_merges);
  out[5] = slots;
  out[6] = std::max(1, most);  // the largest CTA's page list
  out[7] = static_cast<int32_t>(words * 4);
  out[8] = static_cast<int32_t>(num_shared);
  out[9] = shared_max;
  out[10] = static_cast<int32_t>(pieces.size());
  out[11] = layout;
  int32_t* item = out + kPlanHeaderWords;
  int32_t* seg = out + kPlanHeaderWords + num_items * kPlanItemWords + merges.size() +
                 num_shared * kPlanSharedWords;
  int next_seg = 0;
  for (int k : order) {
    item[0] = kPlanKindSegments;
    item[1] = next_seg;
    item[2] = bin_first[k + 1] - bin_first[k];
    item[3] = bin_pages[k];
    for (int j = bin_first[k]; j < bin_first[k + 1]; ++j) {
      const int i = by_bin[j];
      const Piece& pc = pieces[i];
      seg[0] = pc.b;
      seg[1] = lens[pc.b];
      seg[2] = pc.p_begin;
      seg[3] = pc.n;
      seg[4] = piece_slot[i];
      if (npieces[pc.b] == 1 && group_of[pc.b] >= 0) {  // fold the shared partials
        seg[5] = shared_ranges[group_of[pc.b]];
        seg[6] = slot_base[pc.b];
      }
      seg += kPlanSegWords;
      ++next_seg;
    }
    item += kPlanItemWords;
  }
  if (!merges.empty()) memcpy(item, merges.data(), merges.size() * 4);
  item += merges.size();
  write_shared_items(groups, shared_ranges, slot_base, item);
  return PKV_OK;
}

// The work unit U: the smallest whose plan fits in one wave of resident
// CTAs (kResidentPerSm per SM, 8 kv heads each item), starting from
// ceil(P / (2 SMs)), the unit at which the ranges alone would fill that
// wave; when none fits (a batch too large for one wave), the ranges take
// the whole table width.  Sequences of up to R pages get one range; longer
// ones are cut into ceil(p / R) ranges of near-equal size, which the merge
// kernel combines.  Items run in order of the pages their busiest warp
// streams, most first (ranges before packed items on ties).
//
// With shared groups, a member attends only its own pages [k, pages) in
// range items (never packed) and every range writes a partial; the group's
// pages [0, k) become shared-prefix items (ns near-equal ranges per group,
// ns the most that keeps these CTAs within one wave of two per SM) whose CTAs write one
// partial per member; each member's partials sit in consecutive slots,
// shared ranges first, and one merge entry combines them.
int build_core(const int32_t* lens, int batch, int max_blocks, int num_sms,
               const std::vector<SharedGroup>& groups, int32_t* out, size_t out_bytes) {
  const long long Lmax = static_cast<long long>(max_blocks) * kPageSize;
  std::vector<int> pages(batch), start(batch, 0), group_of(batch, -1);
  for (int b = 0; b < batch; ++b) {
    if (lens[b] < 0 || lens[b] > Lmax) return PKV_EINVAL;
    pages[b] = ceil_div(lens[b], kPageSize);
  }
  for (size_t gi = 0; gi < groups.size(); ++gi)
    for (int m = 0; m < groups[gi].members; ++m) {
      start[groups[gi].first + m] = groups[gi].k;
      group_of[groups[gi].first + m] = static_cast<int>(gi);
    }
  // what the per-sequence items attend: own pages; members never packed
  std::vector<int> own(batch), solo;  // solo: pages of the sequences in no group
  solo.reserve(batch);
  long long total = 0;
  for (int b = 0; b < batch; ++b) {
    own[b] = pages[b] - start[b];
    total += own[b];
    if (group_of[b] < 0) solo.push_back(own[b]);
  }
  // shared ranges per group: as many as keep the shared-prefix CTAs within
  // one wave of ctas_per_sm per SM, ranges of at least kMinRangePages pages
  std::vector<int> shared_ranges(groups.size());
  int shared_max = 0;  // pages of the longest shared range
  auto plan_shared_ranges = [&](int ctas_per_sm) {
    int ns_target = 1;
    if (!groups.empty()) {
      const long long per = static_cast<long long>(groups.size()) * kNumKvHeads;
      ns_target = static_cast<int>(
          std::max<long long>(1, (static_cast<long long>(ctas_per_sm) * num_sms) / per));
    }
    shared_max = 0;
    for (size_t gi = 0; gi < groups.size(); ++gi) {
      const int k = groups[gi].k;
      int ns = std::max(1, std::min(ns_target, ceil_div(k, kMinRangePages)));
      ns = std::max(ns, ceil_div(k, kMaxRangePages));  // the kernel's page list
      shared_ranges[gi] = ns;
      shared_max = std::max(shared_max, ceil_div(k, ns));
    }
  };
  // A layer whose segment plan has bins of at least kMinSegBinPages pages
  // runs on the segment kernel (one wave of CTAs of near-equal pages); with
  // smaller bins a segment CTA's life is mostly its prologue and the latency
  // of its first pages, and the per-(item, kv head) kernel below, with more
  // CTAs and deeper per-warp rings, is faster (a ragged 16-layer batch of
  // 2067 pages per layer: 313.7 us with bins of 8 pages against 249.7 us).
  // With shared groups whose shared-prefix CTAs fit one per SM, the segment
  // CTAs are sized to run beside them, one per SM (kPlanLayoutBeside), for
  // any layer size whose bins reach kMinSegBinPages: those CTAs overlap the
  // shared-prefix kernel, so small bins cost little there (64 sequences of
  // 2048 tokens in 16-way groups sharing 1536: 26.6 -> 22.8 us against the
  // per-(item, kv head) plan).
  const bool beside = !groups.empty() &&
      static_cast<long long>(groups.size()) * kNumKvHeads <=
          static_cast<long long>(kSharedBesideCtasPerSm) * num_sms;
  if (beside || total >= static_cast<long long>(kMinSegBinPages) * num_sms) {
    static thread_local Packing packing_buf;
    Packing& packing = packing_buf;
    if (beside) {
      bool fitted = false;
      const int T =
          segment_bin_size(own, start, num_sms, kSegBesideCtasPerSm, total, packing, &fitted);
      if (fitted && T >= kMinSegBinPages) {  // one segment CTA per SM, at most
        plan_shared_ranges(kSharedBesideCtasPerSm);
        return build_segments(lens, batch, max_blocks, T, own, start, group_of, groups,
                              shared_ranges, shared_max, kPlanLayoutBeside, packing, out,
                              out_bytes);
      }
    }
    const int T = total >= static_cast<long long>(kMinSegBinPages) * num_sms
                      ? segment_bin_size(own, start, num_sms, kSegCtasPerSm, total, packing)
                      : 0;
    if (T >= kMinSegBinPages) {
      plan_shared_ranges(kSharedCtasPerSm);
      return build_segments(lens, batch, max_blocks, T, own, start, group_of, groups,
                            shared_ranges, shared_max, kPlanLayoutSequential, packing, out,
                            out_bytes);
    }
  }
  // Below the segment plans, the per-(item, kv head) CTAs run beside the
  // shared-prefix CTAs too when those fit one per SM: an SM holding a
  // shared-prefix CTA has registers for kPerHeadBesideCtasPerSm of them.
  long long wave = static_cast<long long>(kResidentPerSm) * num_sms;  // CTAs
  int layout = kPlanLayoutSequential;
  if (beside) {
    plan_shared_ranges(kSharedBesideCtasPerSm);
    long long shared_ctas = 0;
    for (int ns : shared_ranges) shared_ctas += static_cast<long long>(ns) * kNumKvHeads;
    wave -= (kResidentPerSm - kPerHeadBesideCtasPerSm) * std::min<long long>(shared_ctas, num_sms);
    layout = kPlanLayoutBeside;
  } else {
    plan_shared_ranges(kSharedCtasPerSm);
  }

  auto count = [&](Sizes z) {
    long long items = count_items(solo, z);
    for (int b = 0; b < batch; ++b)
      if (group_of[b] >= 0) items += (own[b] + z.range - 1) / z.range;
    return items;
  };
  const long long u0 = std::max<long long>(1, (total + 2LL * num_sms - 1) / (2LL * num_sms));
  const long long umax = std::max<long long>(u0, (max_blocks + kPlanWarps - 1) / kPlanWarps);
  long long lo = u0, hi = umax;  // smallest u in [u0, umax] that fits, else umax
  while (lo < hi) {
    const long long mid = (lo + hi) / 2;
    if (count(sizes_for(mid, max_blocks)) * kNumKvHeads <= wave) hi = mid;
    else lo = mid + 1;
  }
  const Sizes z = sizes_for(lo, max_blocks);
  const int range = z.range;
  const int pack_max = z.pack_max;


  std::vector<Range> ranges;
  std::vector<int> packed;
  std::vector<int32_t> merges;  // (b, first slot, ranges, 0) per split sequence
  ranges.reserve(batch);
  packed.reserve(batch);
  std::vector<int> slot_base(batch, -1);
  int slots = 0;
  for (int b = 0; b < batch; ++b) {
    const int p = own[b];
    const bool member = group_of[b] >= 0;
    if (!member && p <= pack_max) {
      packed.push_back(b);
    } else if (!member && p <= range) {
      ranges.push_back({b, lens[b], 0, p, -1});
    } else {
      const int ns = member ? shared_ranges[group_of[b]] : 0;
      const int nr = ceil_div(p, range);
      const int base = p / nr, extra = p % nr;
      int begin = start[b];
      for (int r = 0; r < nr; ++r) {
        const int n = base + (r < extra ? 1 : 0);
        ranges.push_back({b, lens[b], begin, n, slots + ns + r});
        begin += n;
      }
      merges.insert(merges.end(), {b, slots, ns + nr, 0});
      slot_base[b] = slots;
      slots += ns + nr;
    }
  }
  // packed sequences by pages, most first (stable); packed ones have at most
  // pack_max <= kPackPages pages
  counting_sort(packed, kPackPages + 1, [&](int b) { return kPackPages - pages[b]; });
  // work items with the pages of their busiest warp, most first, ranges
  // before packed items on ties (stable)
  struct Item {
    int work, kind, index;  // index into ranges or into packed (first of 4)
  };
  std::vector<Item> order;
  order.reserve(ranges.size() + packed.size() / kPlanWarps + 1);
  int max_work = 0;
  for (size_t i = 0; i < ranges.size(); ++i) {
    order.push_back({(ranges[i].n + kPlanWarps - 1) / kPlanWarps, kPlanKindRange,
                     static_cast<int>(i)});
    max_work = std::max(max_work, order.back().work);
  }
  for (size_t i = 0; i < packed.size(); i += kPlanWarps) {
    order.push_back({pages[packed[i]], kPlanKindPacked, static_cast<int>(i)});
    max_work = std::max(max_work, order.back().work);
  }
  counting_sort(order, 2 * (max_work + 1),
                [&](const Item& x) { return 2 * (max_work - x.work) + x.kind; });
  const size_t num_items = order.size();
  const size_t num_merges = merges.size() / kPlanMergeWords;
  size_t num_shared = 0;
  for (int ns : shared_ranges) num_shared += static_cast<size_t>(ns);
  if (num_items > 65535 || num_shared > 65535) return PKV_EUNSUPPORTED;  // grid y limit

  const size_t words = kPlanHeaderWords + num_items * kPlanItemWords + merges.size() +
                       num_shared * kPlanSharedWords;
  if (words * 4 > out_bytes) return PKV_EINVAL;
  memset(out, 0, words * 4);
  out[0] = static_cast<int32_t>(PKV_PLAN_MAGIC);
  out[1] = batch;
  out[2] = max_blocks;
  out[3] = static_cast<int32_t>(num_items);
  out[4] = static_cast<int32_t>(num_merges);
  out[5] = slots;
  out[6] = range;
  out[7] = static_cast<int32_t>(words * 4);
  out[8] = static_cast<int32_t>(num_shared);
  out[9] = shared_max;
  out[11] = layout;
  int32_t* item = out + kPlanHeaderWords;
  for (const Item& o : order) {
    if (o.kind == kPlanKindRange) {
      const Range& r = ranges[o.index];
      item[0] = kPlanKindRange;
      item[1] = r.slot;
      item[2] = r.p_begin;
      item[3] = r.n;
      for (int w = 0; w < kPlanWarps; ++w) {
        item[4 + w] = r.b;
        item[8 + w] = r.L;
      }
    } else {
      item[0] = kPlanKindPacked;
      item[1] = -1;
      for (int w = 0; w < kPlanWarps; ++w) {
        const size_t k = static_cast<size_t>(o.index) + w;
        const bool has = k < packed.size();
        item[4 + w] = has ? packed[k] : -1;
        item[8 + w] = has ? lens[packed[k]] : 0;
      }
    }
    item += kPlanItemWords;
  }
  if (!merges.empty()) memcpy(item, merges.data(), merges.size() * 4);
  item += merges.size();
  write_shared_items(groups, shared_ranges, slot_base, item);
  return PKV_OK;
}

int check_plan_args(const int32_t* lens, int batch, int max_blocks, int num_sms,
                    const int32_t* out, size_t out_bytes) {
  if (lens == nullptr || out == nullptr || batch < 1 || max_blocks < 1 || num_sms < 1)
    return PKV_EINVAL;
  if (reinterpret_cast<uintptr_t>(out) % 16 != 0) return PKV_EALIGN;
  if (out_bytes < plan_bytes(batch, max_blocks)) return PKV_EINVAL;
  return PKV_OK;
}

int build_plan(const int32_t* lens, int batch, int max_blocks, int num_sms, int32_t* out,
               size_t out_bytes) {
  const int rc = check_plan_args(lens, batch, max_blocks, num_sms, out, out_bytes);
  if (rc != PKV_OK) return rc;
  return build_core(lens, batch, max_blocks, num_sms, {}, out, out_bytes);
}

// Groups are found in batch order: a run starts at sequence s and takes the
// next sequences while their tables agree with s's on at least the first
// min_shared_pages entries (each a valid page id) and it has fewer than
// kSharedMembers members; k is the shortest agreement, also kept below
// every member's last page.  A run of one sequence is no group.
int build_plan_shared(const int32_t* lens, const int32_t* block_tables, int batch,
                      int max_blocks, int num_sms, int min_shared_pages, int32_t* out,
                      size_t out_bytes) {
  const int rc = check_plan_args(lens, batch, max_blocks, num_sms, out, out_bytes);
  if (rc != PKV_OK) return rc;
  if (block_tables == nullptr || min_shared_pages < 1) return PKV_EINVAL;
  const long long Lmax = static_cast<long long>(max_blocks) * kPageSize;
  std::vector<int> pages(batch);
  for (int b = 0; b < batch; ++b) {
    if (lens[b] < 0 || lens[b] > Lmax) return PKV_EINVAL;
    pages[b] = ceil_div(lens[b], kPageSize);
  }
  auto row = [&](int b) { return block_tables + static_cast<size_t>(b) * max_blocks; };
  // the length of the common start of two rows, up to c entries (memcmp
  // compares 16 entries at a time, then the last block is searched)
  auto common = [](const int32_t* x, const int32_t* y, int c) {
    constexpr int kBlock = 16;
    int i = 0;
    while (i + kBlock <= c && memcmp(x + i, y + i, kBlock * sizeof(int32_t)) == 0) i += kBlock;
    while (i < c && x[i] == y[i]) ++i;
    return i;
  };
  std::vector<SharedGroup> groups;
  int b = 0;
  while (b < batch) {
    int k = pages[b] - 1;  // the leader's last page stays its own
    // only the leader's valid ids are shared: [0, valid) checked so far
    // (stopped at the first negative id, if any)
    int valid = 0;
    auto valid_prefix = [&](int n) {
      while (valid < n && row(b)[valid] >= 0) ++valid;
      return std::min(valid, n);
    };
    int e = b + 1;
    while (e < batch && e - b < kSharedMembers) {
      const int agree = valid_prefix(common(row(b), row(e), std::min(k, pages[e] - 1)));
      if (agree < min_shared_pages) break;
      k = agree;
      ++e;
    }
    if (e - b >= 2 && k >= min_shared_pages) {
      groups.push_back({b, e - b, k});
      b = e;
    } else {
      ++b;
    }
  }
  return build_core(lens, batch, max_blocks, num_sms, groups, out, out_bytes);
}

}  // namespace pkv

extern "C" PKV_API int pkv_check_tables(const int32_t* block_table, int max_blocks,
                                        const int32_t* seq_lens, int batch, int64_t num_pages,
                                        int page_size, int* bad_seq, int* bad_block) {
  auto fail = [&](int b, int blk) {
    if (bad_seq != nullptr) *bad_seq = b;
    if (bad_block != nullptr) *bad_block = blk;
    return PKV_EINVAL;
  };
  if (block_table == nullptr || seq_lens == nullptr || batch < 0 || max_blocks < 1 ||
      num_pages < 1 || page_size < 1)
    return fail(-1, -1);
  const long long Lmax = static_cast<long long>(max_blocks) * page_size;
  for (int b = 0; b < batch; ++b) {
    const int32_t L = seq_lens[b];
    if (L < 0 || L > Lmax) return fail(b, -1);
    const int live = static_cast<int>((static_cast<long long>(L) + page_size - 1) / page_size);
    const int32_t* row = block_table + static_cast<int64_t>(b) * max_blocks;
    for (int k = 0; k < live; ++k)
      if (row[k] < 0 || row[k] >= num_pages) return fail(b, k);
  }
  if (bad_seq != nullptr) *bad_seq = -1;
  if (bad_block != nullptr) *bad_block = -1;
  return PKV_OK;
}

