// plan.cu - device-side plan builder: q2k -> k2q CSR -> task table.
//
// The pages describe this step as the official CSR builder plus a fused
// task builder whose exact counts and CTA schedule never leave the device
// (NeMo-Automodel PR "feat(minimax-m3) ...", Changelog; API page
// msa_backward_sm100: tiles of 8 queries times the 16 query heads of an index
// head, grouped by
// (batch, index_head, key_block)).  Everything here stays on the device and
// is launched with capacity-bounded grids; exact counts are read from the
// plan header.
//
// Octet groups.  The same CTA sees, per key block, which of its 128 queries
// selected it, so it also finds the block's aligned octets (8 queries) whose
// queries all see the same non-empty block set: their tiles can accumulate
// block after block in one place (the forward's group kernel), and the
// forward's pooled task list leaves out the tasks made only of such queries.
// Two such octets 2i, 2i+1 with the same set form one item.  Items are placed
// by decreasing cost (blocks x octets) so that a round-robin walk over them
// balances.
//
// Count entries.  For index head g, document d (n blocks), key block v and
// query block qb >= v, entry (g, d, v, qb) counts the queries of block qb that
// selected v.  Entries are ordered (g, d, super-block of qb, v, qb) - see
// tri_local - so one exclusive scan gives each entry its place in col, queries
// end up ascending within every bucket, and the task table comes out grouped
// by super-block.  A CTA per (g, d, qb) builds a 128-query bitmap per key
// block in shared memory: popcounts give the counts, prefix popcounts give
// each query's rank, and duplicate slots collapse for free.
#include "common.cuh"
#include "sm100.cuh"

namespace msa {
namespace {

constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;
constexpr int kScanTile = kScanThreads * kScanItems;  // elements per scan CTA
constexpr int kChunkV = 1024;                         // key blocks per bitmap pass

// ------------------------------------------------------------ block scans
template <typename Tv>
__device__ __forceinline__ Tv warp_incl_scan(Tv x) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    Tv y = __shfl_up_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) >= o) x += y;
  }
  return x;
}

// Exclusive scan over the CTA (blockDim.x == 1024); returns the prefix of x
// and writes the CTA total to *total.
template <typename Tv>
__device__ Tv block_excl_scan(Tv x, Tv* total) {
  __shared__ Tv warp_tot[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  Tv inc = warp_incl_scan(x);
  if (lane == 31) warp_tot[w] = inc;
  __syncthreads();
  if (w == 0) {
    Tv v = warp_tot[lane];
    Tv vi = warp_incl_scan(v);
    warp_tot[lane] = vi - v;
    if (lane == 31) *total = vi;
  }
  __syncthreads();
  Tv res = inc - x + (w == 0 ? Tv(0) : warp_tot[w]);
  __syncthreads();
  return res;
}

// ------------------------------------------------------------ documents
__global__ void __launch_bounds__(1024) k_plan_docs(msa_plan p) {
  grid_dep_wait();
  grid_dep_release();
  __shared__ int bad;
  __shared__ int64_t tot_nb, tot_tri;
  const int32_t* offs = p.doc_offsets;
  const int D = p.num_docs;
  int64_t* hdr = p.header;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kHdrWords; ++i) hdr[i] = 0;
    bad = (offs[0] != 0 || int64_t(offs[D]) != p.T);
  }
  for (int64_t i = threadIdx.x; i < p.scan_tmp_len; i += blockDim.x) p.scan_tmp[i] = 0;
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x)
    if (offs[d + 1] <= offs[d]) bad = 1;
  __syncthreads();
  if (bad) {
    if (threadIdx.x == 0) raise_status(hdr, MSA_ERR_BAD_OFFSETS);
    return;
  }
  DocInfo* info = reinterpret_cast<DocInfo*>(p.doc_info);
  int64_t carry_nb = 0, carry_tri = 0;
  for (int base = 0; base < D; base += blockDim.x) {
    const int d = base + threadIdx.x;
    int64_t nb = 0, start = 0, len = 0;
    if (d < D) {
      start = offs[d];
      len = int64_t(offs[d + 1]) - start;
      nb = (len + kBlock - 1) / kBlock;
    }
    const int64_t tri = nb * (nb + 1) / 2;
    const int64_t ex_nb = block_excl_scan<int64_t>(nb, &tot_nb);
    const int64_t ex_tri = block_excl_scan<int64_t>(tri, &tot_tri);
    if (d < D) {
      info[d] = DocInfo{int32_t(start), int32_t(len), int32_t(nb), int32_t(carry_nb + ex_nb)};
      p.doc_tri[d] = carry_tri + ex_tri;
    }
    __syncthreads();
    carry_nb += tot_nb;
    carry_tri += tot_tri;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    p.doc_tri[D] = carry_tri;
    if (4 * carry_tri > p.tri_cap || carry_nb > p.nb_cap) {
      raise_status(hdr, MSA_ERR_CAPACITY);
      return;
    }
    hdr[kHdrNB] = carry_nb;
    hdr[kHdrTriPerG] = carry_tri;
    hdr[kHdrTri] = 4 * carry_tri;
  }
}

// ------------------------------------------------------------ per query block
enum BlockPass { kPassCount = 0, kPassScatter = 1, kPassEmit = 2 };

template <int PASS>
__global__ void __launch_bounds__(128, 6) k_plan_blocks(msa_plan p) {
  grid_dep_wait();
  grid_dep_release();
  __shared__ uint32_t bm[kChunkV][4];
  __shared__ int s_doc, s_skip;
  __shared__ unsigned long long s_pairs;
  __shared__ int s_nsel[16];        // per octet: blocks selected by any of its queries
  __shared__ uint32_t s_bad, s_pdiff;  // octets not uniform; pairs with different sets
  __shared__ uint64_t s_mask[128];     // dense octets: each query's block mask
  __shared__ int64_t s_hist[kMaxItemCost + 1];  // items per cost
  int64_t* hdr = p.header;
  const int64_t NB = hdr[kHdrNB];
  const int g = int(blockIdx.x / p.nb_cap);
  const int64_t gb = int64_t(blockIdx.x % p.nb_cap);
  if (gb >= NB) return;
  const DocInfo* info = reinterpret_cast<const DocInfo*>(p.doc_info);
  if (threadIdx.x == 0) {
    // Read once and broadcast: another CTA may raise the status meanwhile.
    s_skip = plan_failed(hdr) ? 1 : 0;
    int lo = 0, hi = p.num_docs - 1;  // last document whose first block <= gb
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (info[mid].blk_base <= gb) lo = mid; else hi = mid - 1;
    }
    s_doc = lo;
    s_pairs = 0;
    s_bad = 0u;
    s_pdiff = 0u;
  }
  if (threadIdx.x < 16) s_nsel[threadIdx.x] = 0;
  __syncthreads();
  if (s_skip) return;
  const int d = s_doc;
  const DocInfo di = info[d];
  const int64_t n = di.nblk;
  const int64_t qb = gb - di.blk_base;
  const int64_t Zs = p.super_block > 0 ? p.super_block : n;
  const int64_t seg = int64_t(g) * hdr[kHdrTriPerG] + p.doc_tri[d];
  const int r = threadIdx.x;
  const int64_t pos = qb * kBlock + r;
  const bool valid = pos < di.len;
  const int64_t t = di.start + pos;

  int32_t sl[kTopK];
  if (valid) {
    const int4* src = reinterpret_cast<const int4*>(p.q2k + (int64_t(g) * p.T + t) * kTopK);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int4 x = src[i];
      sl[4 * i + 0] = x.x; sl[4 * i + 1] = x.y; sl[4 * i + 2] = x.z; sl[4 * i + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kTopK; ++i) sl[i] = -1;
  }
  if (PASS == kPassCount && valid) {
#pragma unroll
    for (int i = 0; i < kTopK; ++i)
      if (sl[i] < -1 || sl[i] >= n) raise_status(hdr, MSA_ERR_BAD_Q2K);
  }
  // A slot counts once: later duplicates of a value are dropped.
#pragma unroll
  for (int i = 1; i < kTopK; ++i)
#pragma unroll
    for (int j = 0; j < i; ++j)
      if (sl[i] == sl[j]) sl[i] = -1;

  const int64_t lo_q = (qb / Zs) * Zs;       // first query block of this super-block
  const int64_t hi_q = lo_q + Zs < n ? lo_q + Zs : n;
  int64_t pairs = 0;
  // octet scan: thread r looks at octet r % 16 for every eighth key block
  const int oct = r & 15;
  auto octet_rows = [&](int o) -> int {  // valid queries of octet o
    const int64_t rem = int64_t(di.len) - (qb * kBlock + 8 * o);
    return rem <= 0 ? 0 : (rem >= 8 ? 8 : int(rem));
  };
  const uint32_t oct_mask = (1u << octet_rows(oct)) - 1u;
  int my_nsel = 0;
  bool my_bad = false, my_pdiff = false;

  for (int64_t c0 = 0; c0 <= qb; c0 += kChunkV) {
    const int64_t cend = (c0 + kChunkV - 1 < qb) ? c0 + kChunkV - 1 : qb;
    const int span = int(cend - c0 + 1);
    for (int i = threadIdx.x; i < span * 4; i += blockDim.x) (&bm[0][0])[i] = 0u;
    __syncthreads();
    if (valid) {
#pragma unroll
      for (int i = 0; i < kTopK; ++i)
        if (sl[i] >= c0 && sl[i] <= cend) atomicOr(&bm[sl[i] - c0][r >> 5], 1u << (r & 31));
    }
    __syncthreads();
    if (PASS != kPassEmit) {
      for (int v = r >> 4; v < span; v += 8) {
        const uint32_t b0 = (bm[v][oct >> 2] >> ((oct & 3) * 8)) & 0xFFu;
        my_nsel += b0 != 0u;
        my_bad |= b0 != 0u && b0 != oct_mask;
        if (!(oct & 1)) {
          const uint32_t b1 = (bm[v][(oct + 1) >> 2] >> (((oct + 1) & 3) * 8)) & 0xFFu;
          my_pdiff |= (b0 != 0u) != (b1 != 0u);
        }
      }
    }
    if (PASS == kPassCount) {
      for (int64_t v = c0 + threadIdx.x; v <= cend; v += blockDim.x) {
        const uint32_t* b = bm[v - c0];
        p.cnt[seg + tri_local(n, Zs, v, qb)] =
            __popc(b[0]) + __popc(b[1]) + __popc(b[2]) + __popc(b[3]);
      }
    } else if (PASS == kPassScatter) {
      if (valid) {
        // all bucket offsets in flight before the first use
        int32_t dst[kTopK];
#pragma unroll
        for (int i = 0; i < kTopK; ++i) {
          const int64_t v = sl[i];
          dst[i] = (v >= c0 && v <= cend) ? p.off[seg + tri_local(n, Zs, v, qb)] : 0;
        }
        const int w = r >> 5;
#pragma unroll
        for (int i = 0; i < kTopK; ++i) {
          const int64_t v = sl[i];
          if (v < c0 || v > cend) continue;
          const uint32_t* b = bm[v - c0];
          int rank = __popc(b[w] & ((1u << (r & 31)) - 1u));
          for (int k = 0; k < w; ++k) rank += __popc(b[k]);
          p.col[dst[i] + rank] = int32_t(t);
          pairs += (v < qb) ? kBlock : (pos - qb * kBlock + 1);
        }
      }
      // Tasks per sub-bucket: the run of entries (v, qb') for qb' in
      // [max(v, lo_q), hi_q) is contiguous; its head entry owns the tasks.
      for (int64_t v = c0 + threadIdx.x; v <= cend; v += blockDim.x) {
        const int64_t e = seg + tri_local(n, Zs, v, qb);
        const int64_t first = v > lo_q ? v : lo_q;
        if (qb == first) {
          const int64_t last = e + (hi_q - first) - 1;
          const int64_t len = int64_t(p.off[last]) + p.cnt[last] - p.off[e];
          p.tcnt[e] = int32_t((len + kTaskQueries - 1) / kTaskQueries);
        } else {
          p.tcnt[e] = 0;
        }
      }
    } else {  // kPassEmit
      // Head entries (v, first = max(v, lo_q)) own their run's tasks.  The
      // head of v >= lo_q is emitted by the CTA of query block v; the heads
      // of the key blocks before the super-block (v < lo_q, all in query
      // block lo_q) are spread over the super-block's CTAs, v modulo its
      // length, so that no CTA walks all of them.
      const int64_t span = hi_q - lo_q;
      for (int64_t v = c0; v <= cend; ++v) {
        if (v >= lo_q ? v != qb : v % span != qb - lo_q) continue;
        const int64_t first = v > lo_q ? v : lo_q;
        const int64_t e = seg + tri_local(n, Zs, v, first);
        const int64_t last = e + (hi_q - first) - 1;
        const int64_t len = int64_t(p.off[last]) + p.cnt[last] - p.off[e];
        const int nt = p.tcnt[e];
        const int32_t key_start = int32_t(di.start + v * kBlock);
        const int32_t key_len = int32_t(di.len - v * kBlock < kBlock ? di.len - v * kBlock : kBlock);
        for (int i = threadIdx.x; i < nt; i += blockDim.x) {
          const int64_t rem = len - int64_t(i) * kTaskQueries;
          const int32_t nq = int32_t(rem < kTaskQueries ? rem : kTaskQueries);
          int4 task;
          task.x = p.off[e] + i * kTaskQueries;
          task.y = key_start;
          task.z = key_len | (nq << 8) | (g << 12);
          task.w = int32_t(int64_t(g) * p.nb_cap + di.blk_base + v);
          reinterpret_cast<int4*>(p.tasks)[p.toff[e] + i] = task;
          // the forward's pooled list keeps tasks with an ungrouped query
          int32_t tq[kTaskQueries];
#pragma unroll
          for (int k = 0; k < kTaskQueries; ++k) tq[k] = k < nq ? p.col[task.x + k] : -1;
          int keep = 0;
#pragma unroll
          for (int k = 0; k < kTaskQueries; ++k)
            keep |= tq[k] >= 0 && p.grouped[int64_t(g) * p.T + tq[k]] == 0;
          p.fflag[p.toff[e] + i] = keep;
        }
      }
    }
    __syncthreads();
  }
  if (PASS != kPassEmit) {
    if (my_nsel) atomicAdd(&s_nsel[oct], my_nsel);
    if (my_bad) atomicOr(&s_bad, 1u << oct);
    if (my_pdiff) atomicOr(&s_pdiff, 1u << (oct >> 1));
    // dense octets: this query's visible selected blocks as a bit mask
    const bool dense_ok = qb + 1 <= p.dense_blocks;
    // items per cost (complete after the count pass), for the placements
    if (PASS == kPassScatter)
      for (int c = threadIdx.x; c <= kMaxItemCost; c += blockDim.x)
        s_hist[c] = c == 0 ? 0 : hdr[kHdrCost + c];
    if (PASS == kPassScatter && dense_ok) {
      uint64_t m = 0ull;
#pragma unroll
      for (int i = 0; i < kTopK; ++i)
        if (sl[i] >= 0 && sl[i] <= qb) m |= 1ull << sl[i];
      s_mask[r] = m;
    }
    __syncthreads();
    // s_nsel[o]: blocks some query of octet o selected; s_bad bit o: some
    // block selected by only part of its queries
    auto uniform = [&](int o) {
      return octet_rows(o) > 0 && s_nsel[o] > 0 && !((s_bad >> o) & 1u);
    };
    auto dense = [&](int o) {
      return dense_ok && octet_rows(o) > 0 && s_nsel[o] > 0 && ((s_bad >> o) & 1u);
    };
    auto paired = [&](int i) {
      return (uniform(2 * i) && uniform(2 * i + 1) && !((s_pdiff >> i) & 1u)) ||
             (dense(2 * i) && dense(2 * i + 1));
    };
    const int o = r >> 3;
    if (PASS == kPassCount) {
      const bool grp = uniform(o) || dense(o);
      if (valid) p.grouped[int64_t(g) * p.T + t] = grp ? 1 : 0;
      // the pooled path's rows: appended by warp, in no particular order
      const unsigned m = __ballot_sync(0xffffffffu, valid && !grp);
      if (m) {
        const int lane = r & 31;
        unsigned long long base = 0ull;
        if (lane == 0)
          base = atomicAdd(reinterpret_cast<unsigned long long*>(hdr + kHdrRows),
                           (unsigned long long)__popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        if (valid && !grp)
          p.rows[base + __popc(m & ((1u << lane) - 1u))] = int32_t(t) * kKVHeads + g;
      }
    }
    const bool dn = dense(o);
    if ((r & 7) == 0 && (uniform(o) || dn) && !((o & 1) && paired(o >> 1))) {
      const bool hasB = !(o & 1) && paired(o >> 1);
      const int nsel = dn ? int(qb) + 1 : s_nsel[o];
      const int cost = nsel * (hasB ? 2 : 1);
      unsigned long long* cnt = reinterpret_cast<unsigned long long*>(hdr + kHdrCost);
      if (PASS == kPassCount) {
        atomicAdd(cnt + cost, 1ull);
      } else {
        int64_t pos = 0;  // items of higher cost come first
        for (int c = cost + 1; c <= kMaxItemCost; ++c) pos += s_hist[c];
        pos += int64_t(atomicAdd(
            reinterpret_cast<unsigned long long*>(hdr + kHdrCostFill) + cost, 1ull));
        int32_t* it = p.items + pos * kItemWords;
        *reinterpret_cast<int4*>(it) =
            make_int4(int32_t(t), hasB ? int32_t(t + 8) : -1,
                      octet_rows(o) | (hasB ? octet_rows(o + 1) : 0) << 4 | g << 8 |
                          nsel << 12 | (dn ? 1 : 0) << 20,
                      d);
        if (dn) {
          // the masks of the queries of A, then of B (0 past an octet's end)
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const int oo = o + (k >> 3), qi = k & 7;
            const uint64_t m = (k < 8 || hasB) && qi < octet_rows(oo) ? s_mask[8 * oo + qi] : 0ull;
            it[4 + 2 * k] = int32_t(uint32_t(m));
            it[5 + 2 * k] = int32_t(uint32_t(m >> 32));
          }
        } else {
          // this query's visible blocks (distinct after the dedupe), ascending
          int nb = 0;
#pragma unroll
          for (int i = 0; i < kTopK; ++i) {
            if (sl[i] < 0 || sl[i] > qb) continue;
            int rank = 0;
#pragma unroll
            for (int j = 0; j < kTopK; ++j) rank += (sl[j] >= 0 && sl[j] < sl[i]);
            it[4 + rank] = sl[i];
            ++nb;
          }
          for (int k = nb; k < kItemWords - 4; ++k) it[4 + k] = -1;  // the whole payload
        }
      }
    }
    if (PASS == kPassScatter && blockIdx.x == 0 && threadIdx.x == 0) {
      int64_t tot = 0;
      for (int c = 1; c <= kMaxItemCost; ++c) tot += hdr[kHdrCost + c];
      hdr[kHdrItems] = tot;
    }
  }
  if (PASS == kPassScatter) {
    if (pairs) atomicAdd(&s_pairs, (unsigned long long)pairs);
    __syncthreads();
    if (threadIdx.x == 0 && s_pairs)
      atomicAdd(reinterpret_cast<unsigned long long*>(hdr + kHdrPairs),
                s_pairs * (unsigned long long)kHeadsPerGroup);
  }
}

// ------------------------------------------------------------ device scan
// Exclusive scan of in[0, n) -> out in one pass, n read from the device; the
// total goes to *total.  Decoupled look-back (Merrill and Garland,
// "Single-pass Parallel Prefix Scan with Decoupled Look-back", 2016): a CTA
// takes the next tile by ticket, publishes the tile's sum, then adds up the
// published sums of the tiles before it, back to the first tile that has
// published its inclusive prefix, and publishes its own.  Tickets go out in
// the order CTAs start, so a CTA only waits on CTAs that already run; the
// wait is bounded all the same (MSA_ERR_TIMEOUT, and the CTA publishes
// anyway so that later tiles finish).  st[0] is the ticket counter and
// st[1 + j] the status of tile j: zero, or a flag in the top two bits above
// the value.  k_plan_docs zeroes them.  With a compaction target, element j's
// record csrc[j] is also copied to cdst[out[j]] where in[j] != 0.
constexpr unsigned long long kStAgg = 1ull << 62;   // tile sum published
constexpr unsigned long long kStPre = 1ull << 63;   // inclusive prefix published
constexpr unsigned long long kStVal = kStAgg - 1;

__global__ void __launch_bounds__(kScanThreads) k_scan(const int32_t* in, int32_t* out,
                                                       const int64_t* n_ptr, int64_t cap,
                                                       int64_t* total, unsigned long long* st,
                                                       int64_t* hdr, const int4* csrc,
                                                       int4* cdst) {
  grid_dep_wait();
  grid_dep_release();
  __shared__ int64_t tot, excl_sh;
  __shared__ unsigned tile_sh;
  // A failed plan's counts are not to be trusted (an earlier pass stopped
  // early): nothing to scan then.  n never exceeds the arrays' capacity.
  const int64_t n_dev = plan_failed(hdr) ? 0 : *n_ptr;
  const int64_t n = n_dev < 0 ? 0 : (n_dev > cap ? cap : n_dev);
  if (threadIdx.x == 0) tile_sh = atomicAdd(reinterpret_cast<unsigned*>(st), 1u);
  __syncthreads();
  const int64_t tile = tile_sh;
  const int64_t base = tile * kScanTile;
  if (base >= n) {
    if (tile == 0 && threadIdx.x == 0) *total = 0;
    return;
  }
  int32_t v[kScanItems];
  int64_t s = 0;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t j = base + int64_t(threadIdx.x) * kScanItems + i;
    v[i] = j < n ? in[j] : 0;
    s += v[i];
  }
  const int64_t ex = block_excl_scan<int64_t>(s, &tot);
  if (threadIdx.x < 32) {
    // warp 0 looks back over windows of 32 predecessors at a time
    const int lane = threadIdx.x;
    volatile unsigned long long* stv = st + 1;
    int64_t prefix = 0;
    if (tile > 0) {
      if (lane == 0) stv[tile] = kStAgg | (unsigned long long)tot;
      const uint64_t t0 = global_timer_ns();
      for (int64_t top = tile - 1;;) {
        const int64_t k = top - lane;
        // (before tile 0: an inclusive prefix of 0)
        const unsigned long long x =
            k >= 0 ? (unsigned long long)stv[k] : (unsigned long long)kStPre;
        const unsigned ready = __ballot_sync(0xffffffffu, x != 0ull);
        const unsigned pre = __ballot_sync(0xffffffffu, (x & kStPre) != 0ull);
        // lanes up to the nearest inclusive prefix, when all of them are in
        const unsigned need = pre ? (pre & (0u - pre)) * 2u - 1u : 0xffffffffu;
        if ((ready & need) == need) {
          int64_t val = (need >> lane) & 1u ? int64_t(x & kStVal) : 0;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) val += __shfl_xor_sync(0xffffffffu, val, o);
          prefix += val;
          if (pre) break;
          top -= 32;
          continue;
        }
        const bool late = __shfl_sync(0xffffffffu, global_timer_ns() - t0 > kWaitTimeoutNs, 0);
        if (late) {
          if (lane == 0) raise_status(hdr, MSA_ERR_TIMEOUT);
          break;
        }
      }
    }
    if (lane == 0) {
      stv[tile] = kStPre | (unsigned long long)(prefix + tot);
      excl_sh = prefix;
      if (base + kScanTile >= n) *total = prefix + tot;
    }
  }
  __syncthreads();
  int64_t run = excl_sh + ex;
#pragma unroll
  for (int i = 0; i < kScanItems; ++i) {
    const int64_t j = base + int64_t(threadIdx.x) * kScanItems + i;
    if (j < n) {
      out[j] = int32_t(run);
      if (cdst != nullptr && v[i] != 0) cdst[run] = csrc[j];
    }
    run += v[i];
  }
}

// scan k of the plan (0: cnt, 1: tcnt, 2: fflag) uses status region k
__host__ __device__ inline unsigned long long* scan_status(const msa_plan& p, int k) {
  const int64_t region = p.scan_tmp_len / 6;  // (tiles + 1) words of 64 bits each
  return reinterpret_cast<unsigned long long*>(p.scan_tmp) + k * region;
}

cudaError_t scan(const msa_plan& p, int k, const int32_t* in, int32_t* out, const int64_t* n_ptr,
                 int64_t cap, int64_t* total, cudaStream_t s, const int4* csrc = nullptr,
                 int4* cdst = nullptr) {
  const unsigned grid = unsigned((cap + kScanTile - 1) / kScanTile);
  if (grid == 0) return cudaSuccess;
  launch_begin(k == 2 ? "plan_ftasks" : "plan_scan", s);
  const cudaError_t e = launch_k(true, k_scan, dim3(grid), dim3(kScanThreads), 0, s, in, out, n_ptr,
                                 cap, total, scan_status(p, k), p.header, csrc, cdst);
  launch_end(k == 2 ? "plan_ftasks" : "plan_scan", s);
  return e;
}

}  // namespace

cudaError_t launch_plan(const msa_plan& p, cudaStream_t s) {
  // Every kernel may start during its predecessor's tail (launch_k) and
  // waits for it before touching memory; a caller's kernel that never
  // signals counts as signalling when it completes.
  launch_begin("plan_docs", s);
  cudaError_t e = launch_k(true, k_plan_docs, dim3(1), dim3(1024), 0, s, p);
  launch_end("plan_docs", s);
  if (e != cudaSuccess) return e;
  const unsigned grid = unsigned(4 * p.nb_cap);
  launch_begin("plan_count", s);
  e = launch_k(true, k_plan_blocks<kPassCount>, dim3(grid), dim3(128), 0, s, p);
  launch_end("plan_count", s);
  if (e != cudaSuccess) return e;
  e = scan(p, 0, p.cnt, p.off, p.header + kHdrTri, p.tri_cap, p.header + kHdrNnz, s);
  if (e != cudaSuccess) return e;
  launch_begin("plan_scatter", s);
  e = launch_k(true, k_plan_blocks<kPassScatter>, dim3(grid), dim3(128), 0, s, p);
  launch_end("plan_scatter", s);
  if (e != cudaSuccess) return e;
  e = scan(p, 1, p.tcnt, p.toff, p.header + kHdrTri, p.tri_cap, p.header + kHdrTasks, s);
  if (e != cudaSuccess) return e;
  launch_begin("plan_emit", s);
  e = launch_k(true, k_plan_blocks<kPassEmit>, dim3(grid), dim3(128), 0, s, p);
  launch_end("plan_emit", s);
  if (e != cudaSuccess) return e;
  // the forward's pooled list: tasks with fflag set, in task order
  return scan(p, 2, p.fflag, p.fpos, p.header + kHdrTasks, p.task_cap, p.header + kHdrFTasks, s,
              reinterpret_cast<const int4*>(p.tasks), reinterpret_cast<int4*>(p.ftasks));
}

}  // namespace msa
