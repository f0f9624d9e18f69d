// attn_fwd.cu - MSA forward: O [T,64,128] and LSE [T,64].
//
// The method (NeMo-Automodel PR "feat(minimax-m3): add SM100 MSA sparse
// attention with custom backward", section "Design": the flat forward
// O[T,64,128] from the CSR / schedule) is computed KV-parallel: every task is
// one 128-row tile (8 queries x 16 heads of one index head) against one
// 128-key block, so K/V stay resident in shared memory across the tasks of a
// bucket and each tile is a dense 128x128x128 tensor-core contraction.
//
// The up-to-16 partial results of a row (one per selected block) are merged
// without a second pass over the scores.  Each task exponentiates against its
// own tile row maximum m (P = exp(s - m) in (0, 1], fp16 for the P.V product)
// and rescales its partial P.V and row sum by exp(m - M) onto a per-row shift
// M[t,h] shared by all tasks of the row: the Cauchy-Schwarz bound
// scale * |q_th| * max_{selected v} max_{j in v} |k_jg| on every score of the
// row, lowered by a fixed headroom so that a loose bound (a few keys of large
// norm) does not push the sum towards underflow.  The rescaled partials add up
// in fp32 pools with L2 bulk reductions; the finalize divides.  Rows whose sum
// still underflows (the bound more than headroom + 60 octaves above the true
// maximum) are recomputed exactly by a fallback kernel.
//
// Kernels, in launch order:
//   fwd_kmax      per (index head, key block): max key norm
//   fwd_rows      per (token, index head): row shifts M, zero the pools
//   fwd_main      the tensor-core tile loop (TMA + tcgen05 + TMEM)
//   fwd_finalize  O = pool / sum -> bf16, LSE; flags underflowed rows
//   fwd_fallback  exact recomputation of the flagged rows (usually none)
#include "common.cuh"
#include "sm100.cuh"

namespace msa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// A row whose pooled exponential sum is below 2^-60 is recomputed exactly.
constexpr float kUnderflowSum = 8.673617379884035e-19f;

// ------------------------------------------------------------ workspace
// Bytes per element of the O pool (fp32, or bf16 on request).
inline size_t pool_elem_bytes(const msa_plan& p) { return p.o_accum == MSA_O_ACCUM_BF16 ? 2 : 4; }

struct FwdLayout {
  size_t off_m, off_l, off_pool, off_kmax, off_vmax, off_list, total;
};
FwdLayout fwd_layout(const msa_plan& p) {
  FwdLayout L{};
  const int64_t rows = p.T * kQHeads;
  size_t o = 0;
  L.off_m = o;    o = align_up(o + sizeof(float) * rows, 256);
  L.off_l = o;    o = align_up(o + sizeof(float) * rows, 256);
  L.off_pool = o; o = align_up(o + pool_elem_bytes(p) * rows * kHeadDim, 256);
  L.off_kmax = o; o = align_up(o + sizeof(float) * kKVHeads * p.nb_cap, 256);
  L.off_vmax = o; o = align_up(o + sizeof(float) * kKVHeads * p.nb_cap, 256);
  L.off_list = o; o = align_up(o + sizeof(int32_t) * (rows + 1), 256);
  L.total = o;
  return L;
}

// V tiles enter the P.V product as fp16.  A block whose largest |v| exceeds
// 2^15 is scaled by an exact power of two 2^-e first; the epilogue multiplies
// by 2^e.  Returns 2^-e (1 for every ordinary block).
__device__ __forceinline__ float v_scale_in(float vmax) {
  if (!(vmax > 32768.f)) return 1.f;
  const int e = int(ceilf(log2f(vmax * (1.f / 32768.f))));
  return __int_as_float((127 - (e < 126 ? e : 126)) << 23);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ int doc_of_token(const int32_t* offs, int D, int64_t t) {
  int lo = 0, hi = D - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (offs[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// ------------------------------------------------------------ fwd_kmax
// kmax[g * nb_cap + b] = max over the keys j of global block b of |K[j,g]|.
__global__ void __launch_bounds__(128) k_fwd_kmax(msa_plan p, const __nv_bfloat16* K,
                                                  const __nv_bfloat16* V, float* kmax,
                                                  float* vmax, int32_t* list) {
  __shared__ float red[4][4], redv[4][4];
  if (blockIdx.x == 0 && threadIdx.x == 0) list[0] = 0;  // fallback row count
  const int64_t NB = p.header[kHdrNB];
  const int64_t gb = blockIdx.x;
  if (gb >= NB || plan_failed(p.header)) return;
  const DocInfo* info = reinterpret_cast<const DocInfo*>(p.doc_info);
  int lo = 0, hi = p.num_docs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (info[mid].blk_base <= gb) lo = mid; else hi = mid - 1;
  }
  const DocInfo di = info[lo];
  const int64_t kb = (gb - di.blk_base) * kBlock;
  const int r = threadIdx.x;
  float nrm[4] = {0.f, 0.f, 0.f, 0.f}, vm[4] = {0.f, 0.f, 0.f, 0.f};
  if (kb + r < di.len) {
    const int64_t j = di.start + kb + r;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint4* src = reinterpret_cast<const uint4*>(K + (j * kKVHeads + g) * kHeadDim);
      const uint4* vsrc = reinterpret_cast<const uint4*>(V + (j * kKVHeads + g) * kHeadDim);
      float s = 0.f, m = 0.f;
#pragma unroll 4
      for (int c = 0; c < 16; ++c) {
        const uint4 x = src[c];
        const uint4 y = vsrc[c];
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        const uint32_t u[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
          s = fmaf(a, a, s);
          s = fmaf(b, b, s);
          m = fmaxf(m, fmaxf(fabsf(bf16_lo(u[e])), fabsf(bf16_hi(u[e]))));
        }
      }
      nrm[g] = sqrtf(s);
      vm[g] = m;
    }
  }
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float x = nrm[g], y = vm[g];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
      y = fmaxf(y, __shfl_xor_sync(0xffffffffu, y, o));
    }
    if ((r & 31) == 0) {
      red[g][r >> 5] = x;
      redv[g][r >> 5] = y;
    }
  }
  __syncthreads();
  if (r < 4) {
    const float m = fmaxf(fmaxf(red[r][0], red[r][1]), fmaxf(red[r][2], red[r][3]));
    // Round up by a few ulps so the bound survives the rounding of the
    // tensor-core dot products.
    kmax[int64_t(r) * p.nb_cap + gb] = m * 1.0001f;
    vmax[int64_t(r) * p.nb_cap + gb] =
        fmaxf(fmaxf(redv[r][0], redv[r][1]), fmaxf(redv[r][2], redv[r][3]));
  }
}

// ------------------------------------------------------------ fwd_rows
// One warp per (token, index head): the shift M2 of each of the 16 heads'
// rows (-inf when the row sees no key), and zero the row's pool and sum.
//
// The Cauchy-Schwarz bound B = c2 * |q_th| * kmax_sel (log2 units) is never
// below the row's true maximum m, but may sit far above it (a few keys of
// large norm).  The shift is placed H below it, M2 = B - H, so that the row's
// pooled sum 2^(m - M2) * (...) underflows only when B - m > H + 60.  A
// partial is then scaled by at most 2^H, so the pool holds at most
// 2^H * 2^11 * vmax_sel (2048 keys, P <= 1): H = 64, lowered for rows whose
// selected blocks hold |v| above 2^48, keeps that below 2^124.
constexpr float kShiftHeadroom = 64.f;
__global__ void __launch_bounds__(256) k_fwd_rows(msa_plan p, const __nv_bfloat16* Q,
                                                  const float* kmax, const float* vmax,
                                                  float c2, float* M2, float* lsum,
                                                  uint8_t* pool, int pool_esz) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (wid >= p.T * kKVHeads || plan_failed(p.header)) return;
  const int64_t t = wid >> 2;
  const int g = int(wid & 3);
  const int d = doc_of_token(p.doc_offsets, p.num_docs, t);
  const DocInfo di = reinterpret_cast<const DocInfo*>(p.doc_info)[d];
  const int64_t qb = (t - di.start) / kBlock;
  float km = -1.f, vm = 0.f;
  if (lane < kTopK) {
    const int32_t v = p.q2k[(int64_t(g) * p.T + t) * kTopK + lane];
    if (v >= 0 && v <= qb) {
      km = kmax[int64_t(g) * p.nb_cap + di.blk_base + v];
      vm = vmax[int64_t(g) * p.nb_cap + di.blk_base + v];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
    vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
  }
  // vm may be inf or nan (non-finite V): no headroom then.
  const float headroom =
      (vm <= 281474976710656.f) ? kShiftHeadroom
                                : (vm < INFINITY ? fmaxf(0.f, 112.f - ceilf(log2f(vm))) : 0.f);
  // 16 heads x 128 dims = 4 KB of Q: lanes 0-15 take head 2i, 16-31 head 2i+1.
  const __nv_bfloat16* qrow = Q + (t * kQHeads + g * kHeadsPerGroup) * kHeadDim;
  uint8_t* prow = pool + (t * kQHeads + g * kHeadsPerGroup) * kHeadDim * pool_esz;
  const int half = lane >> 4, sub = lane & 15;
#pragma unroll 2
  for (int i = 0; i < 8; ++i) {
    const int hh = 2 * i + half;
    const uint4 x = reinterpret_cast<const uint4*>(qrow + hh * kHeadDim)[sub];
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
      s = fmaf(a, a, s);
      s = fmaf(b, b, s);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (sub == 0) {
      const int64_t row = t * kQHeads + g * kHeadsPerGroup + hh;
      M2[row] = km < 0.f ? -INFINITY : c2 * sqrtf(s) * km - headroom;
      lsum[row] = 0.f;
    }
  }
  uint4* z = reinterpret_cast<uint4*>(prow);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const int n16 = kHeadsPerGroup * kHeadDim * pool_esz / 16;
#pragma unroll 4
  for (int i = lane; i < n16; i += 32) z[i] = zero;
}

// ------------------------------------------------------------ fwd_main
// Warp roles (480 threads):
//   0     TMA producer: K/V per block run, Q per task (two stages)
//   1     MMA issuer (TMEM owner): S = Q K^T, O_part = P V with P read from TMEM
//   2-9   softmax (thread = tile row = TMEM lane): row max, P = exp(s - m) as
//         fp16 into the stage's P columns, row sum; warps 2-5 take the even
//         tasks (TMEM stage 0), warps 6-9 the odd ones (stage 1)
//   10-13 epilogue (thread = tile row): O_part * exp(m - M) staged in shared
//         memory and added to the fp32 pool by bulk tensor reductions (four
//         2 KB boxes per query, issued by one lane per warp); row sums by
//         atomics
//   14    V tile bf16 -> fp16 (power-of-two scaled when |v| is large)
// TMEM: S in two stages, P (fp16) of each stage in columns of its own, one
// O_part stage (see kTmP0, kTmO).
constexpr int kFwdThreads = 480;
constexpr uint32_t kTileBytes = 32768;
constexpr uint32_t kSmK = 0, kSmV = 32768, kSmQ = 65536, kSmStage = 131072;
// Epilogue staging: per query of the tile, four 2 KB boxes (16 heads x 32
// columns, fp32, 128-byte swizzle) - the boxes of the pool's tensor map.
constexpr uint32_t kStageBytes = kTaskQueries * 8192;
constexpr uint32_t kFwdSmem = kSmStage + kStageBytes + 1024;

// TMEM columns: S in two stages [0,128) and [128,256); P of stage st (fp16
// pairs) in [256 + 64 st, 320 + 64 st); one O_part stage [384,512).  P has
// columns of its own so that S(t+2) can overwrite S(t) as soon as the
// softmax has read it, without waiting for P(t).V.
constexpr uint32_t kTmP0 = 256, kTmO = 384;

struct FwdBars {
  uint64_t kv_full, kv_empty, v_ready, q_full[2], q_empty[2], s_full[2], s_free[2], p_full[2],
      pv_done[2], rs_free[2], o_full, o_free, fin;
};

struct FwdParams {
  msa_plan plan;
  const float* M2;
  const float* vmax;
  void* pool;
  float* lsum;
  float c2;
};

// Task i of the CTA's walk: chunks of kFwdChunk consecutive tasks go round-robin
// over the CTAs, so all CTAs advance through the task list together.
// Tasks per chunk of the CTA walk (a compile-time power of two: the walk's
// index arithmetic runs on the MMA issuer's critical path).
constexpr int kFwdChunk = 16;
__device__ __forceinline__ int64_t cta_task(int64_t i) {
  return (int64_t(blockIdx.x) + (i / kFwdChunk) * gridDim.x) * kFwdChunk + (i % kFwdChunk);
}
__device__ __forceinline__ int64_t cta_task_count(int64_t ntasks) {
  constexpr int chunk = kFwdChunk;
  const int64_t nchunks = (ntasks + chunk - 1) / chunk;
  if (int64_t(blockIdx.x) >= nchunks) return 0;
  const int64_t mine = (nchunks - 1 - blockIdx.x) / gridDim.x + 1;  // chunks of this CTA
  const int64_t last_chunk = blockIdx.x + (mine - 1) * gridDim.x;
  return (mine - 1) * chunk + (ntasks - last_chunk * chunk < chunk ? ntasks - last_chunk * chunk
                                                                    : chunk);
}
// Task record i of this CTA's walk; past the end, the last one (every
// caller guards its uses by the index).  Only the address depends on the
// index test, never the loaded value, so nothing waits for the load until
// the record is used.  With no tasks, entry 0 of the (allocated) table.
__device__ __forceinline__ int4 task_rec(const int4* tasks, int64_t i, int64_t n) {
  return tasks[n > 0 ? cta_task(i < n ? i : n - 1) : 0];
}
__device__ __forceinline__ int32_t task_token(const int32_t* col, const TaskView& tv, int qi) {
  return col[tv.col_begin + (qi < tv.nq ? qi : tv.nq - 1)];
}

// Softmax of one tile row held in TMEM columns [cs, cs + 128) of the
// thread's lane: keys after jmax are excluded when MASK (diagonal and partial
// blocks, padded queries with jmax = -1).
template <bool MASK>
__device__ __forceinline__ float tile_row_max(uint32_t cs, int jmax) {
  float m[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) m[e] = -INFINITY;
  auto reduce = [&](const uint32_t (&r)[16], int lim) {  // lim = jmax - first column
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      float x0 = __uint_as_float(r[j]), x1 = __uint_as_float(r[j + 1]);
      if (MASK) {
        x0 = j <= lim ? x0 : -INFINITY;
        x1 = j + 1 <= lim ? x1 : -INFINITY;
      }
      m[(j >> 1) & 3] = fmax3(m[(j >> 1) & 3], x0, x1);
    }
  };
  uint32_t r0[16], r1[16];
  tmem_ld16(cs, r0);
  tmem_ld_wait();
  reg_fence16(r0);
  // 16-column chunks 2i (r0) and 2i+1 (r1); the next chunk loads while the
  // current one is reduced
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    tmem_ld16(cs + 32 * i + 16, r1);
    reduce(r0, jmax - 32 * i);
    tmem_ld_wait();
    reg_fence16(r1);
    if (i < 3) tmem_ld16(cs + 32 * i + 32, r0);
    reduce(r1, jmax - 32 * i - 16);
    if (i < 3) {
      tmem_ld_wait();
      reg_fence16(r0);
    }
  }
  return fmaxf(fmax3(m[0], m[1], m[2]), m[3]);
}

// P = 2^(s c2 - mxc) written as fp16 pairs over the columns already read
// (columns [cs + 8c, cs + 8c + 8) after reading [cs + 16c, cs + 16c + 16));
// the next 16 columns are loaded while the current ones are exponentiated.
// Returns the row sum of the fp32 values.
template <bool MASK>
__device__ __forceinline__ float tile_row_exp(uint32_t cs, uint32_t cp, int jmax, float c2,
                                             float mxc) {
  const uint64_t cc = f2_pack(__float_as_uint(c2), __float_as_uint(c2));
  const uint64_t nm = f2_pack(__float_as_uint(-mxc), __float_as_uint(-mxc));
  uint64_t ls[4] = {0ull, 0ull, 0ull, 0ull};
  auto expo = [&](const uint32_t (&r)[16], int lim, uint32_t dst) {
    uint32_t pk[8];
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      const uint64_t x2 = f2_fma(f2_pack(r[j], r[j + 1]), cc, nm);
      float p0 = fast_exp2(f2_lo(x2)), p1 = fast_exp2(f2_hi(x2));
      if (MASK) {
        p0 = j <= lim ? p0 : 0.f;
        p1 = j + 1 <= lim ? p1 : 0.f;
      }
      ls[(j >> 1) & 3] =
          f2_add(ls[(j >> 1) & 3], f2_pack(__float_as_uint(p0), __float_as_uint(p1)));
      pk[j >> 1] = pack_f16x2(p0, p1);
    }
    tmem_st8_nc(dst, pk);
  };
  uint32_t r0[16], r1[16];
  tmem_ld16(cs, r0);
  tmem_ld_wait();
  reg_fence16(r0);
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    tmem_ld16(cs + 32 * i + 16, r1);
    expo(r0, jmax - 32 * i, cp + 16 * i);
    tmem_ld_wait();
    reg_fence16(r1);
    if (i < 3) tmem_ld16(cs + 32 * i + 32, r0);
    expo(r1, jmax - 32 * i - 16, cp + 16 * i + 8);
    if (i < 3) {
      tmem_ld_wait();
      reg_fence16(r0);
    }
  }
  const uint64_t s2 = f2_add(f2_add(ls[0], ls[1]), f2_add(ls[2], ls[3]));
  return f2_lo(s2) + f2_hi(s2);
}

// MMA issuer of k_fwd_main (one thread).  A function of its own so its few
// live values stay in registers whatever the other roles need.
__device__ __noinline__ void fwd_mma_role(FwdBars& bars, uint32_t tmem, uint32_t sbase,
                                          const int4* tasks, int64_t my_n,
                                          volatile int* abort_flag) {
  constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);  // Q . K^T   (bf16)
  constexpr uint32_t idPV = idesc_f16_f32(128, 128, 0, 1);  // P . V     (fp16, P in TMEM)
  auto wait = [&](uint64_t& bar, uint32_t ph) {
    return mbar_wait(smem_u32(&bar), ph, abort_flag);
  };
  // Descriptors are built once; a k-step only adds a constant to the
  // start-address field (addresses stay below 256 KB, so the 14-bit field
  // never carries).
  const uint64_t kK = sdesc_sw128(sbase + kSmK, 16u, 1024u);     // K, K-major
  const uint64_t mV = sdesc_sw128(sbase + kSmV, 16384u, 1024u);  // V (fp16), MN-major
  const uint64_t kQ0 = sdesc_sw128(sbase + kSmQ, 16u, 1024u);
  constexpr uint64_t kStage = kTileBytes >> 4;
  auto kstep = [](int kk) { return uint64_t((kk >> 2) * 1024 + (kk & 3) * 2); };
  auto mstep = [](int kk) { return uint64_t(kk) * 128u; };
  int64_t kv_loads = 0;
  bool ok = true, need_v = false;
  // S(it) goes to stage it&1, which the softmax of task it-2 must have read.
  auto issue_S = [&](int64_t it) -> bool {
    const int st = int(it & 1);
    if (!wait(bars.q_full[st], uint32_t((it >> 1) & 1))) return false;
    if (it >= 2 && !wait(bars.s_free[st], uint32_t(((it >> 1) - 1) & 1))) return false;
    tc_fence_after();
    const uint64_t bq = kQ0 + uint64_t(st) * kStage;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ss(tmem + st * 128, bq + kstep(kk), kK + kstep(kk), idS, kk > 0);
    umma_commit(smem_u32(&bars.s_full[st]));
    umma_commit(smem_u32(&bars.q_empty[st]));
    return true;
  };
  auto wait_kv = [&]() -> bool {
    if (!wait(bars.kv_full, uint32_t(kv_loads & 1))) return false;
    ++kv_loads;
    need_v = true;
    return true;
  };
  int cur_kv = task_rec(tasks, 0, my_n).w;
  int next_kv = task_rec(tasks, 1, my_n).w;
  ok = wait_kv() && issue_S(0);
  for (int64_t it = 0; ok && it < my_n; ++it) {
    const int st = int(it & 1);
    const int next2_kv = task_rec(tasks, it + 2, my_n).w;
    const bool same = (it + 1 < my_n) && next_kv == cur_kv;
    if (same && !issue_S(it + 1)) break;
    if (!wait(bars.p_full[st], uint32_t((it >> 1) & 1))) break;
    // one O_part stage: the epilogue must have read O_part(it-1)
    if (it >= 1 && !wait(bars.o_free, uint32_t((it - 1) & 1))) break;
    if (need_v) {
      if (!wait(bars.v_ready, uint32_t((kv_loads - 1) & 1))) break;
      need_v = false;
    }
    tc_fence_after();
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ts(tmem + kTmO, tmem + kTmP0 + st * 64 + kk * 8, mV + mstep(kk), idPV, kk > 0);
    umma_commit(smem_u32(&bars.o_full));
    umma_commit(smem_u32(&bars.pv_done[st]));
    if (it + 1 < my_n && !same) {
      umma_commit(smem_u32(&bars.kv_empty));
      cur_kv = next_kv;
      if (!wait_kv() || !issue_S(it + 1)) break;
    }
    next_kv = next2_kv;
  }
  // Make sure no MMA is still running before TMEM is released.
  umma_commit(smem_u32(&bars.fin));
  mbar_wait_drain(smem_u32(&bars.fin), 0);
}

// POOL_BF16: the O pool is bf16 (boxes of 64 columns) instead of fp32 (boxes
// of 32 columns).
template <bool POOL_BF16>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_fwd_main(const __grid_constant__ FwdParams prm, const __grid_constant__ CUtensorMap mapQ,
               const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
               const __grid_constant__ CUtensorMap mapPool) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, skip_sh;
  __shared__ float s_alpha[2][128], s_lrow[2][128];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const msa_plan& p = prm.plan;
  volatile int* abort_flag = &abort_sh;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    skip_sh = plan_failed(p.header) ? 1 : 0;
    mbar_init(smem_u32(&bars.kv_full), 1);
    mbar_init(smem_u32(&bars.kv_empty), 1);
    mbar_init(smem_u32(&bars.v_ready), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.q_full[i]), 1);
      mbar_init(smem_u32(&bars.q_empty[i]), 1);
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.s_free[i]), 128);
      mbar_init(smem_u32(&bars.p_full[i]), 128);
      mbar_init(smem_u32(&bars.pv_done[i]), 1);
      mbar_init(smem_u32(&bars.rs_free[i]), 128);
    }
    mbar_init(smem_u32(&bars.o_full), 1);
    mbar_init(smem_u32(&bars.o_free), 128);
    mbar_init(smem_u32(&bars.fin), 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_base_sh), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_sh;
  const int64_t ntasks = skip_sh ? 0 : p.header[kHdrTasks];
  const int64_t my_n = cta_task_count(ntasks);
  const int4* tasks = reinterpret_cast<const int4*>(p.tasks);

  if (warp == 0) {
    // ---------------- TMA producer (records and tokens prefetched one task ahead)
    if (lane == 0 && my_n > 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      int prev_kv = -1;
      int64_t kv_loads = 0, it = 0;
      int4 rec = task_rec(tasks, 0, my_n), rec1 = task_rec(tasks, 1, my_n);
      int32_t tok[kTaskQueries];
      {
        const TaskView tv = decode_task(rec);
#pragma unroll
        for (int qi = 0; qi < kTaskQueries; ++qi) tok[qi] = task_token(p.col, tv, qi);
      }
      for (; it < my_n; ++it) {
        const TaskView tv = decode_task(rec);
        const int4 rec2 = task_rec(tasks, it + 2, my_n);
        int32_t tok1[kTaskQueries];
        {
          const TaskView tv1 = decode_task(rec1);
#pragma unroll
          for (int qi = 0; qi < kTaskQueries; ++qi)
            tok1[qi] = it + 1 < my_n ? task_token(p.col, tv1, qi) : 0;
        }
        if (tv.sub != prev_kv) {
          if (kv_loads > 0 &&
              !mbar_wait(smem_u32(&bars.kv_empty), uint32_t((kv_loads - 1) & 1), abort_flag))
            break;
          const uint32_t b = smem_u32(&bars.kv_full);
          mbar_arrive_expect_tx(b, 2 * kTileBytes);
          tma_load_3d(sbase + kSmK, &mapK, b, 0, tv.g, tv.key_start);
          tma_load_3d(sbase + kSmK + 16384, &mapK, b, 64, tv.g, tv.key_start);
          tma_load_3d(sbase + kSmV, &mapV, b, 0, tv.g, tv.key_start);
          tma_load_3d(sbase + kSmV + 16384, &mapV, b, 64, tv.g, tv.key_start);
          ++kv_loads;
          prev_kv = tv.sub;
        }
        const int st = int(it & 1);
        if (it >= 2 &&
            !mbar_wait(smem_u32(&bars.q_empty[st]), uint32_t(((it >> 1) - 1) & 1), abort_flag))
          break;
        const uint32_t b = smem_u32(&bars.q_full[st]);
        mbar_arrive_expect_tx(b, kTileBytes);
        const uint32_t dst = sbase + kSmQ + st * kTileBytes;
#pragma unroll
        for (int qi = 0; qi < kTaskQueries; ++qi) {
          const int y = tok[qi] * kQHeads + tv.g * kHeadsPerGroup;
          tma_load_2d(dst + qi * 2048, &mapQ, b, 0, y);
          tma_load_2d(dst + 16384 + qi * 2048, &mapQ, b, 64, y);
        }
        rec = rec1;
        rec1 = rec2;
#pragma unroll
        for (int qi = 0; qi < kTaskQueries; ++qi) tok[qi] = tok1[qi];
      }
      if (*abort_flag) {  // let armed copies land before the CTA exits
        if (kv_loads > 0) mbar_wait_drain(smem_u32(&bars.kv_full), uint32_t((kv_loads - 1) & 1));
        for (int64_t j = (it >= 2 ? it - 2 : 0); j < it; ++j)
          mbar_wait_drain(smem_u32(&bars.q_full[j & 1]), uint32_t((j >> 1) & 1));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0 && my_n > 0) fwd_mma_role(bars, tmem, sbase, tasks, my_n, abort_flag);
  } else if (warp == 14) {
    // ---------------- V tile bf16 -> fp16 (scaled by an exact power of two)
    if (my_n > 0) {
      int prev_kv = -1;
      int64_t kv_loads = 0;
      for (int64_t it = 0; it < my_n; ++it) {
        const int kv = task_rec(tasks, it, my_n).w;
        if (kv == prev_kv) continue;
        prev_kv = kv;
        const float sc = v_scale_in(prm.vmax[kv]);
        if (!mbar_wait_warp(smem_u32(&bars.kv_full), uint32_t(kv_loads & 1), abort_flag)) break;
        ++kv_loads;
        for (int i = lane; i < 2048; i += 32) {
          const uint32_t a = sbase + kSmV + i * 16;
          const uint4 x = ld_shared_v4(a);
          st_shared_v4(a, pack_f16x2(bf16_lo(x.x) * sc, bf16_hi(x.x) * sc),
                       pack_f16x2(bf16_lo(x.y) * sc, bf16_hi(x.y) * sc),
                       pack_f16x2(bf16_lo(x.z) * sc, bf16_hi(x.z) * sc),
                       pack_f16x2(bf16_lo(x.w) * sc, bf16_hi(x.w) * sc));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars.v_ready));
      }
    }
  } else if (warp < 10) {
    // ---------------- softmax (warps 2-5: even tasks, 6-9: odd tasks)
    const int quad = warp & 3;
    const int par = (warp - 2) >> 2;
    const int row = quad * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    const int qi = row >> 4, hh = row & 15;
    // Row data of this warpgroup's next task (it+2) is loaded while task it
    // runs, in two steps so no load result is consumed right after it is
    // issued: the row's token at the top of task it, its shift M after the
    // exponentials.
    int4 rec1 = task_rec(tasks, par + 2, my_n);
    int jmax_c = -1;
    float m2_c = 0.f;
    if (par < my_n) {
      const TaskView tv = decode_task(task_rec(tasks, par, my_n));
      const int32_t tok = task_token(p.col, tv, qi);
      jmax_c = qi < tv.nq ? min(tok - tv.key_start, tv.key_len - 1) : -1;
      m2_c = prm.M2[int64_t(tok) * kQHeads + tv.g * kHeadsPerGroup + hh];
    }
    for (int64_t it = par; it < my_n; it += 2) {
      const int st = int(it & 1);
      const int jmax = jmax_c;
      const float m2 = m2_c;
      const int4 rec2 = task_rec(tasks, it + 4, my_n);
      // (loads of the next task's row data are unconditional - rec1 is a
      // valid record even past the end - so nothing waits for them here)
      const int32_t ntok = task_token(p.col, decode_task(rec1), qi);
      if (!mbar_wait_warp(smem_u32(&bars.s_full[st]), uint32_t((it >> 1) & 1), abort_flag)) break;
      tc_fence_after();
      const uint32_t cs = tmem + lane_base + st * 128;
      // A warp whose 32 rows all see the whole key block (every tile that is
      // not on a document's diagonal or last partial block) skips the masks.
      const bool full = __all_sync(0xffffffffu, jmax == kBlock - 1);
      // pass 1: the tile row's maximum over visible keys (raw scores)
      const float mx = full ? tile_row_max<false>(cs, jmax) : tile_row_max<true>(cs, jmax);
      const float mxc = (jmax >= 0) ? mx * prm.c2 : 0.f;
      // pass 2: P = exp(s - m) as fp16 pairs into this stage's P columns
      // (P.V of task it-2 must have read them), row sum of the fp32 values
      if (it >= 2 &&
          !mbar_wait_warp(smem_u32(&bars.pv_done[st]), uint32_t(((it >> 1) - 1) & 1), abort_flag))
        break;
      const uint32_t cp = tmem + lane_base + kTmP0 + st * 64;
      const float lsum = full ? tile_row_exp<false>(cs, cp, jmax, prm.c2, mxc)
                              : tile_row_exp<true>(cs, cp, jmax, prm.c2, mxc);
      // S(it) is fully read: S(it+2) may overwrite the stage
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.s_free[st]));
      {  // this warpgroup's next task
        const TaskView tn = decode_task(rec1);
        jmax_c = qi < tn.nq ? min(ntok - tn.key_start, tn.key_len - 1) : -1;
        m2_c = prm.M2[int64_t(ntok) * kQHeads + tn.g * kHeadsPerGroup + hh];
      }
      // the epilogue of task it-2 has read this stage's row scalars
      if (it >= 2 &&
          !mbar_wait_warp(smem_u32(&bars.rs_free[st]), uint32_t(((it >> 1) - 1) & 1), abort_flag))
        break;
      s_alpha[st][row] = jmax >= 0 ? fast_exp2(mxc - m2) : 0.f;
      s_lrow[st][row] = lsum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.p_full[st]));
      rec1 = rec2;
    }
  } else {
    // ---------------- epilogue (warps 10-13)
    // Each thread owns one tile row.  A warp's 32 rows are the 16 heads of
    // two queries; the warp stages them in the 128-byte-swizzled box layout of
    // the pool's tensor map (conflict-free: the eight rows of a store phase
    // hit eight different 16-byte bank groups) and one lane adds them to the
    // pool with four (fp32 pool) or two (bf16 pool) bulk tensor reductions
    // per query.
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    const int qi = row >> 4, hh = row & 15;
    const uint32_t stage_q = sbase + kSmStage + uint32_t(qi) * 8192u;
    const uint32_t stage_row = stage_q + uint32_t(hh) * 128u;
    const uint32_t swz = uint32_t(hh & 7);
    if (lane == 0 && my_n > 0) tma_prefetch_desc(&mapPool);
    int4 rec = task_rec(tasks, 0, my_n), rec1 = task_rec(tasks, 1, my_n);
    // the row's token and the block's V scale are loaded one task ahead
    int32_t tok_c = my_n > 0 ? task_token(p.col, decode_task(rec), qi) : 0;
    float vmax_c = my_n > 0 ? prm.vmax[rec.w] : 0.f;
    for (int64_t it = 0; it < my_n; ++it) {
      const int st = int(it & 1);
      const TaskView tv = decode_task(rec);
      const int4 rec2 = task_rec(tasks, it + 2, my_n);
      const int32_t tok = tok_c;
      const float vmx = vmax_c;
      tok_c = task_token(p.col, decode_task(rec1), qi);  // rec1: a valid record
      vmax_c = prm.vmax[rec1.w];
      const bool valid = qi < tv.nq;
      const int64_t grow = int64_t(tok) * kQHeads + tv.g * kHeadsPerGroup + hh;
      if (!mbar_wait_warp(smem_u32(&bars.o_full), uint32_t(it & 1), abort_flag)) break;
      // p_full(it) completed before o_full(it); waiting on it makes the
      // softmax's row scalars visible here.
      if (!mbar_wait_warp(smem_u32(&bars.p_full[st]), uint32_t((it >> 1) & 1), abort_flag)) break;
      tc_fence_after();
      const float alpha = s_alpha[st][row];
      const float lrow = s_lrow[st][row];
      mbar_arrive(smem_u32(&bars.rs_free[st]));
      const float mul = alpha / v_scale_in(vmx);
      // Boxes 0-1 (columns 0-63) and 2-3 (columns 64-127) of the warp's two
      // queries go out as two bulk groups, so the bulk engine reads one pair
      // while the warp stages the other: before a pair is overwritten, the
      // previous task's group for it must have been read (wait_group.read 1
      // leaves only the most recent group pending).
      const uint32_t obase = tmem + lane_base + kTmO;
      const int32_t tok_hi = __shfl_sync(0xffffffffu, tok, 16);
      auto stage_box = [&](int cq, const uint32_t (&v)[32]) {
#pragma unroll
        for (int u = 0; u < 8; ++u)
          st_shared_v4(stage_row + uint32_t(cq) * 2048u + ((uint32_t(u) ^ swz) << 4),
                       __float_as_uint(__uint_as_float(v[4 * u + 0]) * mul),
                       __float_as_uint(__uint_as_float(v[4 * u + 1]) * mul),
                       __float_as_uint(__uint_as_float(v[4 * u + 2]) * mul),
                       __float_as_uint(__uint_as_float(v[4 * u + 3]) * mul));
      };
      auto issue_pair = [&](int cq0) {  // boxes cq0, cq0 + 1 of both queries
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int qj = 2 * quad + j;
          if (qj < tv.nq) {
            const int y = (j ? tok_hi : tok) * kQHeads + tv.g * kHeadsPerGroup;
#pragma unroll
            for (int cq = cq0; cq < cq0 + 2; ++cq)
              tma_reduce_add_2d(&mapPool, sbase + kSmStage + uint32_t(qj) * 8192u + cq * 2048u,
                                cq * 32, y);
          }
        }
        bulk_commit();
      };
      // bf16 pool: box b holds columns [64b, 64b + 64) of the 16 rows; chunk u
      // of a row (columns 64b + 8u ...) comes from a (u < 4) or b (u >= 4).
      auto stage_box16 = [&](int b, const uint32_t (&a)[32], const uint32_t (&c)[32]) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t (&v)[32] = u < 4 ? a : c;
          const int k = (u & 3) * 8;
          st_shared_v4(stage_row + uint32_t(b) * 2048u + ((uint32_t(u) ^ swz) << 4),
                       pack_bf16x2(__uint_as_float(v[k + 0]) * mul, __uint_as_float(v[k + 1]) * mul),
                       pack_bf16x2(__uint_as_float(v[k + 2]) * mul, __uint_as_float(v[k + 3]) * mul),
                       pack_bf16x2(__uint_as_float(v[k + 4]) * mul, __uint_as_float(v[k + 5]) * mul),
                       pack_bf16x2(__uint_as_float(v[k + 6]) * mul, __uint_as_float(v[k + 7]) * mul));
        }
      };
      auto issue_box16 = [&](int b) {  // box b of both queries
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int qj = 2 * quad + j;
          if (qj < tv.nq) {
            const int y = (j ? tok_hi : tok) * kQHeads + tv.g * kHeadsPerGroup;
            tma_reduce_add_2d(&mapPool, sbase + kSmStage + uint32_t(qj) * 8192u + b * 2048u,
                              b * 64, y);
          }
        }
        bulk_commit();
      };
      uint32_t v0[32], v1[32];
      tmem_ld32(obase, v0);
      tmem_ld32(obase + 32, v1);
      if (lane == 0) bulk_wait_read1();  // previous task's boxes 0-1 read
      __syncwarp();
      tmem_ld_wait();
      reg_fence32(v0);
      reg_fence32(v1);
      if constexpr (POOL_BF16) {
        stage_box16(0, v0, v1);
      } else {
        stage_box(0, v0);
        stage_box(1, v1);
      }
      tmem_ld32(obase + 64, v0);
      tmem_ld32(obase + 96, v1);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if constexpr (POOL_BF16)
          issue_box16(0);
        else
          issue_pair(0);
      }
      __syncwarp();
      tmem_ld_wait();
      reg_fence32(v0);
      reg_fence32(v1);
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.o_free));  // O_part read: the next P.V may overwrite it
      if (lane == 0) bulk_wait_read1();  // previous task's boxes 2-3 read
      __syncwarp();
      if constexpr (POOL_BF16) {
        stage_box16(1, v0, v1);
      } else {
        stage_box(2, v0);
        stage_box(3, v1);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if constexpr (POOL_BF16)
          issue_box16(1);
        else
          issue_pair(2);
      }
      if (valid) atomicAdd(prm.lsum + grow, alpha * lrow);
      rec = rec1;
      rec1 = rec2;
    }
    if (lane == 0) bulk_wait0();  // bulk reductions complete before the CTA exits
  }

  // ---------------- teardown
  if (threadIdx.x == 0 && abort_sh) raise_status(p.header, MSA_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ fwd_finalize
// O = pool / sum -> bf16 and LSE = (M + log2 sum) ln 2.  Each warp finishes
// eight rows per step (16 lanes x 8 elements per row), all loads issued
// before any use.  Rows whose sum underflowed are listed for the fallback.
constexpr int kFinRowsPerWarp = 8;
template <bool POOL_BF16>
__global__ void __launch_bounds__(256) k_fwd_finalize(msa_plan p, const float* M2,
                                                      const float* lsum, const void* pool,
                                                      __nv_bfloat16* O, float* lse,
                                                      int32_t* list) {
  if (plan_failed(p.header)) return;
  const int lane = threadIdx.x & 31, sub = lane & 15;
  const int64_t rows = p.T * kQHeads;
  const int64_t nwarps = int64_t(gridDim.x) * blockDim.x / 32;
  for (int64_t r0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32 * kFinRowsPerWarp;
       r0 < rows; r0 += nwarps * kFinRowsPerWarp) {
    float4 a[4], b[4];
    uint4 h[4];  // bf16 pool: the 8 elements, widened after all loads
    float m2[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = r0 + 2 * i + (lane >> 4);
      if (row < rows) {
        if constexpr (POOL_BF16) {
          h[i] = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(pool) +
                                                row * kHeadDim)[sub];
        } else {
          const float4* src =
              reinterpret_cast<const float4*>(static_cast<const float*>(pool) + row * kHeadDim) +
              2 * sub;
          a[i] = src[0];
          b[i] = src[1];
        }
        m2[i] = M2[row];
        l[i] = lsum[row];
      } else {
        m2[i] = -INFINITY;
        l[i] = 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = r0 + 2 * i + (lane >> 4);
      if (row >= rows) continue;
      uint4 out = make_uint4(0u, 0u, 0u, 0u);
      float L = -INFINITY;
      if (m2[i] != -INFINITY) {
        if (!(l[i] >= kUnderflowSum) || !isfinite(l[i])) {
          if (sub == 0) {
            const int32_t k = atomicAdd(list, 1);
            list[1 + k] = int32_t(row);
          }
          continue;  // the fallback kernel writes this row
        }
        const float inv = 1.f / l[i];
        if constexpr (POOL_BF16) {
          a[i] = make_float4(bf16_lo(h[i].x), bf16_hi(h[i].x), bf16_lo(h[i].y), bf16_hi(h[i].y));
          b[i] = make_float4(bf16_lo(h[i].z), bf16_hi(h[i].z), bf16_lo(h[i].w), bf16_hi(h[i].w));
        }
        out = make_uint4(pack_bf16x2(a[i].x * inv, a[i].y * inv), pack_bf16x2(a[i].z * inv, a[i].w * inv),
                         pack_bf16x2(b[i].x * inv, b[i].y * inv), pack_bf16x2(b[i].z * inv, b[i].w * inv));
        L = (m2[i] + __log2f(l[i])) * kLn2;
      }
      reinterpret_cast<uint4*>(O + row * kHeadDim)[sub] = out;
      if (sub == 0) lse[row] = L;
    }
  }
}

// ------------------------------------------------------------ fwd_fallback
// Exact recomputation (online softmax in fp32, CUDA cores) of the flagged
// rows.  One warp per row; lane l owns dims 4l..4l+3.
__global__ void __launch_bounds__(256) k_fwd_fallback(msa_plan p, const __nv_bfloat16* Q,
                                                      const __nv_bfloat16* K,
                                                      const __nv_bfloat16* V, float c2,
                                                      const int32_t* list, __nv_bfloat16* O,
                                                      float* lse) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = int64_t(gridDim.x) * blockDim.x / 32;
  const int32_t n = list[0];
  for (int64_t w = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32; w < n; w += nwarps) {
    const int64_t row = list[1 + w];
    const int64_t t = row / kQHeads;
    const int h = int(row % kQHeads), g = h / kHeadsPerGroup;
    const int d = doc_of_token(p.doc_offsets, p.num_docs, t);
    const DocInfo di = reinterpret_cast<const DocInfo*>(p.doc_info)[d];
    const int64_t pos = t - di.start, qb = pos / kBlock;
    const uint2 qv = reinterpret_cast<const uint2*>(Q + row * kHeadDim)[lane];
    const float q0 = bf16_lo(qv.x), q1 = bf16_hi(qv.x), q2 = bf16_lo(qv.y), q3 = bf16_hi(qv.y);
    float m = -INFINITY, l = 0.f, a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    const int32_t* sel = p.q2k + (int64_t(g) * p.T + t) * kTopK;
    for (int i = 0; i < kTopK; ++i) {
      const int32_t v = sel[i];
      if (v < 0 || v > qb) continue;
      bool dup = false;
      for (int j = 0; j < i; ++j) dup |= (sel[j] == v);
      if (dup) continue;
      const int64_t jend = (v == qb) ? pos : int64_t(v) * kBlock + kBlock - 1;
      for (int64_t jj = int64_t(v) * kBlock; jj <= jend; ++jj) {
        const int64_t key = di.start + jj;
        const uint2 kv = reinterpret_cast<const uint2*>(K + (key * kKVHeads + g) * kHeadDim)[lane];
        float s = q0 * bf16_lo(kv.x) + q1 * bf16_hi(kv.x) + q2 * bf16_lo(kv.y) + q3 * bf16_hi(kv.y);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        s *= c2;
        const float mn = fmaxf(m, s);
        const float corr = exp2f(m - mn), e = exp2f(s - mn);
        const uint2 vv = reinterpret_cast<const uint2*>(V + (key * kKVHeads + g) * kHeadDim)[lane];
        l = l * corr + e;
        a0 = a0 * corr + e * bf16_lo(vv.x);
        a1 = a1 * corr + e * bf16_hi(vv.x);
        a2 = a2 * corr + e * bf16_lo(vv.y);
        a3 = a3 * corr + e * bf16_hi(vv.y);
        m = mn;
      }
    }
    uint2 out = make_uint2(0u, 0u);
    float L = -INFINITY;
    if (l > 0.f) {
      const float inv = 1.f / l;
      out.x = pack_bf16x2(a0 * inv, a1 * inv);
      out.y = pack_bf16x2(a2 * inv, a3 * inv);
      L = (m + log2f(l)) * kLn2;
    }
    reinterpret_cast<uint2*>(O + row * kHeadDim)[lane] = out;
    if (lane == 0) lse[row] = L;
  }
}

}  // namespace

// ------------------------------------------------------------ host side
CUresult make_map_rows(CUtensorMap* m, const void* base, int64_t rows);      // msa_api.cu
CUresult make_map_kv(CUtensorMap* m, const void* base, int64_t T);           // msa_api.cu
CUresult make_map_pool32(CUtensorMap* m, const void* base, int64_t rows);    // msa_api.cu
CUresult make_map_pool16(CUtensorMap* m, const void* base, int64_t rows);    // msa_api.cu
int device_sm_count();                                                       // msa_api.cu

size_t forward_workspace_bytes(const msa_plan& p) { return fwd_layout(p).total; }

cudaError_t launch_forward(const msa_plan& p, const void* q, const void* k, const void* v,
                           float scale, void* o, float* lse, void* ws, cudaStream_t s) {
  const FwdLayout L = fwd_layout(p);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* M2 = reinterpret_cast<float*>(w + L.off_m);
  float* lsum = reinterpret_cast<float*>(w + L.off_l);
  float* vmax = reinterpret_cast<float*>(w + L.off_vmax);
  uint8_t* pool = w + L.off_pool;
  const bool pool16 = p.o_accum == MSA_O_ACCUM_BF16;
  float* kmax = reinterpret_cast<float*>(w + L.off_kmax);
  int32_t* list = reinterpret_cast<int32_t*>(w + L.off_list);
  const float c2 = scale * kLog2e;

  CUtensorMap mQ, mK, mV, mPool;
  if (make_map_rows(&mQ, q, p.T * kQHeads) != CUDA_SUCCESS ||
      make_map_kv(&mK, k, p.T) != CUDA_SUCCESS || make_map_kv(&mV, v, p.T) != CUDA_SUCCESS ||
      (pool16 ? make_map_pool16(&mPool, pool, p.T * kQHeads)
              : make_map_pool32(&mPool, pool, p.T * kQHeads)) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  cudaError_t e;
  launch_begin("fwd_kmax", s);
  k_fwd_kmax<<<unsigned(p.nb_cap), 128, 0, s>>>(p, static_cast<const __nv_bfloat16*>(k),
                                                static_cast<const __nv_bfloat16*>(v), kmax, vmax,
                                                list);
  launch_end("fwd_kmax", s);
  const int64_t warps = p.T * kKVHeads;
  launch_begin("fwd_rows", s);
  k_fwd_rows<<<unsigned((warps + 7) / 8), 256, 0, s>>>(
      p, static_cast<const __nv_bfloat16*>(q), kmax, vmax, c2, M2, lsum, pool,
      int(pool_elem_bytes(p)));
  launch_end("fwd_rows", s);

  static bool attr_set[2] = {false, false};
  if (!attr_set[pool16]) {
    e = cudaFuncSetAttribute(pool16 ? k_fwd_main<true> : k_fwd_main<false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmem);
    if (e != cudaSuccess) return e;
    attr_set[pool16] = true;
  }
  FwdParams prm{p, M2, vmax, pool, lsum, c2};
  const unsigned grid = unsigned(device_sm_count());
  launch_begin("fwd_main", s);
  if (pool16)
    k_fwd_main<true><<<grid, kFwdThreads, kFwdSmem, s>>>(prm, mQ, mK, mV, mPool);
  else
    k_fwd_main<false><<<grid, kFwdThreads, kFwdSmem, s>>>(prm, mQ, mK, mV, mPool);
  launch_end("fwd_main", s);
  launch_begin("fwd_finalize", s);
  if (pool16)
    k_fwd_finalize<true><<<grid * 16, 256, 0, s>>>(p, M2, lsum, pool,
                                                   static_cast<__nv_bfloat16*>(o), lse, list);
  else
    k_fwd_finalize<false><<<grid * 16, 256, 0, s>>>(p, M2, lsum, pool,
                                                    static_cast<__nv_bfloat16*>(o), lse, list);
  launch_end("fwd_finalize", s);
  launch_begin("fwd_fallback", s);
  k_fwd_fallback<<<unsigned(device_sm_count() * 4), 256, 0, s>>>(
      p, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), c2, list, static_cast<__nv_bfloat16*>(o), lse);
  launch_end("fwd_fallback", s);
  return cudaGetLastError();
}

}  // namespace msa
