// attn_fwd.cu - MSA forward: O [T,64,128] and LSE [T,64].
//
// The method (NeMo-Automodel PR "feat(minimax-m3): add SM100 MSA sparse
// attention with custom backward", section "Design": the flat forward
// O[T,64,128] from the CSR / schedule) is computed on 128-row tiles (8
// queries x 16 heads of one index head) against one 128-key block, each a
// dense 128x128x128 tensor-core contraction.
//
// Every row (token, head) gets a shift M shared by all its tiles: the
// Cauchy-Schwarz bound scale * |q_th| * max_{selected v} max_{j in v} |k_jg|
// on its scores, lowered by a fixed headroom so that a loose bound (a few
// keys of large norm) does not push the sum towards underflow.  Tiles
// exponentiate against it, P = exp(s - M) as bf16 (same exponent range as
// fp32), so the partials P.V and row sums of a row add up plainly, in any
// order, without a second pass over the scores and without rescaling.
//
// Two schedules share that arithmetic:
//   * grouped octets (8 consecutive tokens of a document whose tokens see the
//     same blocks; the plan finds them): one CTA takes the octet (with a
//     second one of the same blocks) and walks its blocks, the tile's O
//     accumulating in tensor memory - written out once, no pool;
//   * every other query: KV-parallel tasks, K/V resident in shared memory
//     across the tasks of a bucket; the partials go to an fp32 pool with L2
//     bulk reductions, and the finalize divides.
// Rows whose sum still underflows (the bound more than headroom + 60
// octaves above the true maximum) are recomputed exactly by a fallback.
//
// Kernels, in launch order:
//   fwd_kmax      per (index head, key block): max key norm, max |v|
//   fwd_v16       V as fp16 for the P.V products
//   fwd_group     grouped octets: block walk with O in tensor memory
//   fwd_rows      per ungrouped (token, index head): row shifts M, zero the pool
//   fwd_main      the pooled task loop (TMA + tcgen05 + TMEM)
//   fwd_finalize  pooled rows: O = pool / sum -> bf16, LSE; flags underflow
//   fwd_fallback  exact recomputation of the flagged rows (usually none)
#include "common.cuh"
#include "sm100.cuh"

namespace msa {

#ifdef MSA_TEST_STARVE
// Test-only build: the kernel whose CTA 0 leaves out its first Q tile (1:
// fwd_group, 2: fwd_main, 0: none), so that a bounded wait runs out and the
// call reports MSA_ERR_TIMEOUT.  Set by msa_test_starve.
__device__ int g_starve_fwd;
cudaError_t test_set_starve_fwd(int which) {
  return cudaMemcpyToSymbol(g_starve_fwd, &which, sizeof which);
}
#endif

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// A row whose pooled exponential sum is below 2^-60 is recomputed exactly.
constexpr float kUnderflowSum = 8.673617379884035e-19f;

// ------------------------------------------------------------ workspace

struct FwdLayout {
  size_t off_m, off_l, off_pool, off_kmax, off_vmax, off_list, off_v16, off_vscale, total;
};
FwdLayout fwd_layout(const msa_plan& p) {
  FwdLayout L{};
  const int64_t rows = p.T * kQHeads;
  size_t o = 0;
  L.off_m = o;    o = align_up(o + sizeof(float) * rows, 256);
  L.off_l = o;    o = align_up(o + sizeof(float) * rows, 256);
  L.off_pool = o; o = align_up(o + sizeof(float) * rows * kHeadDim, 256);
  L.off_kmax = o; o = align_up(o + sizeof(float) * kKVHeads * p.nb_cap, 256);
  L.off_vmax = o; o = align_up(o + sizeof(float) * kKVHeads * p.nb_cap, 256);
  L.off_list = o; o = align_up(o + sizeof(int32_t) * (rows + 1), 256);
  L.off_v16 = o;  o = align_up(o + sizeof(uint16_t) * p.T * kKVHeads * kHeadDim, 256);
  L.off_vscale = o; o = align_up(o + sizeof(float) * kKVHeads, 256);
  L.total = o;
  return L;
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
// One CTA per global key block b (its 128 keys x 4 KV heads are 128 KB of K
// and of V, contiguous):
//   kmax[g * nb_cap + b] = max over the block's keys j of |K[j,g]|,
//   vmax[g * nb_cap + b] = max over them of |V[j,g,d]|,
// and V[j,g] converted to fp16 into the forward's copy, unscaled (fwd_v16
// rescales the copy in the rare case that some |v| exceeds 2^15).  Sixteen
// lanes read one 256-byte (key, head) row, so every warp access is 512
// contiguous bytes; a thread's rows all belong to one head.
constexpr int kKmaxThreads = 512;
__global__ void __launch_bounds__(kKmaxThreads) k_fwd_kmax(msa_plan p, const __nv_bfloat16* K,
                                                           const __nv_bfloat16* V, float* kmax,
                                                           float* vmax, int32_t* list,
                                                           uint4* v16) {
  grid_dep_wait();
  grid_dep_release();
  constexpr int kRowsPerPass = kKmaxThreads / 16;              // 32 rows per pass
  constexpr int kPasses = kBlock * kKVHeads / kRowsPerPass;    // 16 passes
  __shared__ float hk[kRowsPerPass], hv[kRowsPerPass];
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
  const int nkeys = int(di.len - kb < kBlock ? di.len - kb : kBlock);
  const int c = threadIdx.x & 15;        // 16-byte chunk of the row
  const int r0 = threadIdx.x >> 4;       // row slot: rows r0 + 32 pass, all of head r0 % 4
  const int64_t base = (di.start + kb) * kKVHeads * (kHeadDim / 8);  // block's first chunk
  const uint4* ksrc = reinterpret_cast<const uint4*>(K) + base;
  const uint4* vsrc = reinterpret_cast<const uint4*>(V) + base;
  uint4* vdst = v16 + base;
  // all sixteen passes' loads in flight before any use
  float nrm = 0.f, vm = 0.f;
  {
    uint4 x[kPasses];
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) {
      const int row = ps * kRowsPerPass + r0;  // key row / 4, head row % 4
      x[ps] = (row >> 2) < nkeys ? ksrc[int64_t(row) * 16 + c] : make_uint4(0u, 0u, 0u, 0u);
    }
    float ss[kPasses];
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) {
      const uint32_t w[4] = {x[ps].x, x[ps].y, x[ps].z, x[ps].w};
      float a = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
        a = fmaf(lo, lo, fmaf(hi, hi, a));
      }
      ss[ps] = a;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1)
#pragma unroll
      for (int ps = 0; ps < kPasses; ++ps) ss[ps] += __shfl_xor_sync(0xffffffffu, ss[ps], o);
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) nrm = fmaxf(nrm, sqrtf(ss[ps]));
  }
  {
    uint4 y[kPasses];
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) {
      const int row = ps * kRowsPerPass + r0;
      y[ps] = (row >> 2) < nkeys ? vsrc[int64_t(row) * 16 + c] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int ps = 0; ps < kPasses; ++ps) {
      const int row = ps * kRowsPerPass + r0;
      const uint32_t u[4] = {y[ps].x, y[ps].y, y[ps].z, y[ps].w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        vm = fmaxf(vm, fmaxf(fabsf(bf16_lo(u[e])), fabsf(bf16_hi(u[e]))));
      if ((row >> 2) < nkeys)
        vdst[int64_t(row) * 16 + c] = make_uint4(pack_f16x2(bf16_lo(u[0]), bf16_hi(u[0])),
                                                 pack_f16x2(bf16_lo(u[1]), bf16_hi(u[1])),
                                                 pack_f16x2(bf16_lo(u[2]), bf16_hi(u[2])),
                                                 pack_f16x2(bf16_lo(u[3]), bf16_hi(u[3])));
    }
  }
  // per row slot r0 (head r0 % 4): the max over the 16 lanes, then over the
  // eight slots of each head
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, o));
  if (c == 0) {
    hk[r0] = nrm;
    hv[r0] = vm;
  }
  __syncthreads();
  if (threadIdx.x < kKVHeads) {
    const int h = threadIdx.x;
    float m = 0.f, mv = 0.f;
    for (int q = h; q < kRowsPerPass; q += kKVHeads) {
      m = fmaxf(m, hk[q]);
      mv = fmaxf(mv, hv[q]);
    }
    // Round up by a few ulps so the bound survives the rounding of the
    // tensor-core dot products.
    kmax[int64_t(h) * p.nb_cap + gb] = m * 1.0001f;
    vmax[int64_t(h) * p.nb_cap + gb] = mv;
  }
}

// ------------------------------------------------------------ fwd_v16
// V enters the P.V products as fp16 (P is fp16, and one tensor-core product
// takes one operand type).  fp16 holds |v| up to 65504, so every value of KV
// head g is scaled by 2^-e_g, e_g the smallest exponent that brings g's
// largest |v| to at most 2^15 (0 for ordinary data); the kernels multiply O
// by vscale[g] = 2^e_g.  fwd_kmax already wrote the unscaled copy, which is
// exact and final when every e_g is 0; otherwise this kernel rewrites it.
__device__ __forceinline__ float v_scale_in(float vmax) {
  if (!(vmax > 32768.f)) return 1.f;
  const int e = int(ceilf(log2f(vmax * (1.f / 32768.f))));
  return __int_as_float((127 - (e < 126 ? e : 126)) << 23);
}
__global__ void __launch_bounds__(256) k_fwd_v16(msa_plan p, const __nv_bfloat16* V,
                                                 const float* vmax, uint4* v16, float* vscale) {
  grid_dep_wait();
  grid_dep_release();
  __shared__ float red[8][4];
  if (plan_failed(p.header)) return;
  const int64_t NB = p.header[kHdrNB];
  float m[4] = {0.f, 0.f, 0.f, 0.f};
  for (int64_t i = threadIdx.x; i < NB; i += blockDim.x)
#pragma unroll
    for (int g = 0; g < 4; ++g) m[g] = fmaxf(m[g], vmax[int64_t(g) * p.nb_cap + i]);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m[g] = fmaxf(m[g], __shfl_xor_sync(0xffffffffu, m[g], o));
    if (lane == 0) red[w][g] = m[g];
  }
  __syncthreads();
  float sc[4];
  bool scaled = false;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float x = red[0][g];
    for (int k = 1; k < int(blockDim.x >> 5); ++k) x = fmaxf(x, red[k][g]);
    sc[g] = v_scale_in(x);
    scaled |= sc[g] != 1.f;
  }
  if (blockIdx.x == 0 && threadIdx.x < 4) vscale[threadIdx.x] = 1.f / sc[threadIdx.x];
  if (!scaled) return;
  const int64_t n = p.T * kKVHeads * kHeadDim / 8;  // 16-byte chunks, 16 per (token, head)
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const float f = sc[(i >> 4) & 3];
    const uint4 x = reinterpret_cast<const uint4*>(V)[i];
    v16[i] = make_uint4(pack_f16x2(bf16_lo(x.x) * f, bf16_hi(x.x) * f),
                        pack_f16x2(bf16_lo(x.y) * f, bf16_hi(x.y) * f),
                        pack_f16x2(bf16_lo(x.z) * f, bf16_hi(x.z) * f),
                        pack_f16x2(bf16_lo(x.w) * f, bf16_hi(x.w) * f));
  }
}

// ------------------------------------------------------------ row shifts
// The Cauchy-Schwarz bound B = c2 * |q_th| * kmax_sel (log2 units) is never
// below the row's true maximum m, but may sit far above it (a few keys of
// large norm).  The shift is placed H below it, M2 = B - H, so that the row's
// pooled sum 2^(m - M2) * (...) underflows only when B - m > H + 60.  A
// partial is then scaled by at most 2^H, so the pool holds at most
// 2^H * 2^11 * vmax_sel (2048 keys, P <= 1): H = 64, lowered for rows whose
// selected blocks hold |v| above 2^48, keeps that below 2^124.
constexpr float kShiftHeadroom = 64.f;
// km: max key norm over the row's visible selected blocks (< 0: none);
// vm: their max |v| (may be inf or nan for non-finite V: no headroom then).
__device__ __forceinline__ float row_shift(float c2, float qnorm, float km, float vm) {
  const float headroom =
      (vm <= 281474976710656.f) ? kShiftHeadroom
                                : (vm < INFINITY ? fmaxf(0.f, 112.f - ceilf(log2f(vm))) : 0.f);
  return km < 0.f ? -INFINITY : c2 * qnorm * km - headroom;
}

// ------------------------------------------------------------ fwd_rows
// One warp per ungrouped (token, index head), from the plan's list of the
// pooled path's rows: the shift M2 of each of the 16 heads' rows (-inf when
// the row sees no key), and zero the row's pool and sum.  Grouped rows are
// the group kernel's alone.
__global__ void __launch_bounds__(256) k_fwd_rows(msa_plan p, const __nv_bfloat16* Q,
                                                  const float* kmax, const float* vmax,
                                                  float c2, float* M2, float* lsum,
                                                  float* pool) {
  grid_dep_wait();
  grid_dep_release();
  if (plan_failed(p.header)) return;
  const int lane = threadIdx.x & 31;
  // a warp per entry of the plan's list of pooled rows (4 t + g)
  const int64_t nrows = p.header[kHdrRows];
  const int64_t nw = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t wi = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; wi < nrows;
       wi += nw) {
    const int32_t ent = p.rows[wi];
    const int64_t t = ent >> 2;
    const int g = ent & 3;
    // 16 heads x 128 dims = 4 KB of Q: lanes 0-15 take head 2i, 16-31 head
    // 2i+1.  The Q loads and the pool's zeroing go out first; the lookups of
    // the row's blocks (document, q2k, kmax) run while they are in flight.
    const __nv_bfloat16* qrow = Q + (t * kQHeads + g * kHeadsPerGroup) * kHeadDim;
    float* prow = pool + (t * kQHeads + g * kHeadsPerGroup) * kHeadDim;
    const int half = lane >> 4, sub = lane & 15;
    uint4 x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      x[i] = reinterpret_cast<const uint4*>(qrow + (2 * i + half) * kHeadDim)[sub];
    float4* z = reinterpret_cast<float4*>(prow);
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = lane; i < kHeadsPerGroup * kHeadDim / 4; i += 32) z[i] = zero;
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
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int hh = 2 * i + half;
      const uint32_t w[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
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
        M2[row] = row_shift(c2, sqrtf(s), km, vm);
        lsum[row] = 0.f;
      }
    }
  }
}

// ------------------------------------------------------------ shared pieces
constexpr uint32_t kTileBytes = 32768;

// Maximum raw score of one tile row held in TMEM columns [cs, cs + 128) of
// the thread's lane over its visible keys (keys after jmax are excluded when
// MASK: diagonal and partial blocks, rows with jmax = -1); 16 columns load
// while the previous 16 are reduced.
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

// P = 2^(s c2 - mref) of one tile row held in TMEM columns [cs, cs + 128),
// written as fp16 pairs to columns [cp, cp + 64): columns [cp + 8c,
// cp + 8c + 8) after reading [cs + 16c, cs + 16c + 16), the next 16 columns
// loading while the current ones are exponentiated (cp may equal cs: a chunk
// only overwrites columns already read).  mref is at or above the row's
// scores less 8 octaves, so P <= 2^8 fits fp16 with an 11-bit significand.
// Keys after jmax get P = 0 when MASK.  Returns the row sum of the fp32
// values.
template <bool MASK>
__device__ __forceinline__ float tile_row_exp(uint32_t cs, uint32_t cp, int jmax, float c2,
                                             float mref) {
  const uint64_t cc = f2_pack(__float_as_uint(c2), __float_as_uint(c2));
  const uint64_t nm = f2_pack(__float_as_uint(-mref), __float_as_uint(-mref));
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

// Loads the 8 queries x 16 heads of one index head (two 16 KB column halves,
// 128-byte swizzled) into a tile: one {64 cols, 16 rows} box per query and half.
__device__ __forceinline__ void load_q_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            const int32_t (&tok)[kTaskQueries], int g) {
#pragma unroll
  for (int qi = 0; qi < kTaskQueries; ++qi) {
    const int y = tok[qi] * kQHeads + g * kHeadsPerGroup;
    tma_load_2d(dst + qi * 2048, map, bar, 0, y);
    tma_load_2d(dst + 16384 + qi * 2048, map, bar, 64, y);
  }
}
// K and V of one key block of KV head g (keys past T read as zero).
__device__ __forceinline__ void load_kv_tiles(uint32_t dk, uint32_t dv, const CUtensorMap* mk,
                                              const CUtensorMap* mv, uint32_t bar, int g,
                                              int key_start) {
  tma_load_3d(dk, mk, bar, 0, g, key_start);
  tma_load_3d(dk + 16384, mk, bar, 64, g, key_start);
  tma_load_3d(dv, mv, bar, 0, g, key_start);
  tma_load_3d(dv + 16384, mv, bar, 64, g, key_start);
}

// ------------------------------------------------------------ fwd_main
// The pooled tasks (the plan's forward list: tasks with at least one
// ungrouped query; grouped queries in them are masked).
// Warp roles (448 threads):
//   0     TMA producer: K/V per block run, Q per task (two stages)
//   1     MMA issuer (TMEM owner): S = Q K^T, O_part = P V with P read from TMEM
//   2-9   softmax (thread = tile row = TMEM lane): row max m over the tile,
//         P = exp(s - m) as fp16 (the maximum is exactly 1) into the stage's
//         P columns, row sum; warps 2-5 take the even tasks (TMEM stage 0),
//         warps 6-9 the odd ones (stage 1)
//   10-13 epilogue (thread = tile row): O_part * exp(m - M) staged in shared
//         memory and added to the fp32 pool by bulk tensor reductions (four
//         2 KB boxes per query, issued by one lane per warp); row sums by
//         atomics
// TMEM: S in two stages, P (fp16) of each stage in columns of its own, one
// O_part stage (see kTmP0, kTmO).  V tiles come from the forward's fp16 copy.
constexpr int kFwdThreads = 448;
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
  uint64_t kv_full, kv_empty, q_full[2], q_empty[2], s_full[2], s_free[2], p_full[2],
      pv_done[2], rs_free[2], o_full, o_free, fin;
};

struct FwdParams {
  msa_plan plan;
  const float* M2;
  const float* kmax;
  const float* vmax;
  float* pool;
  float* lsum;
  int32_t* list;  // fallback rows: [0] count, then rows
  __nv_bfloat16* O;
  float* lse;
  const float* vscale;  // per KV head: 2^e of the fp16 V copy
  float c2;
};

// Tasks per chunk of the CTA walk (TaskWalk: full rounds of chunks go
// round-robin over the CTAs, the rest is split evenly).
constexpr int kFwdChunk = 16;
// Task record i of this CTA's walk; past the end, the last one (every
// caller guards its uses by the index).  Only the address depends on the
// index test, never the loaded value, so nothing waits for the load until
// the record is used.  With no tasks, entry 0 of the (allocated) table.
__device__ __forceinline__ int4 task_rec(const int4* tasks, int64_t i, const TaskWalk& w) {
  return tasks[w.n > 0 ? walk_task<kFwdChunk>(w, i < w.n ? i : w.n - 1) : 0];
}
__device__ __forceinline__ int32_t task_token(const int32_t* col, const TaskView& tv, int qi) {
  return col[tv.col_begin + (qi < tv.nq ? qi : tv.nq - 1)];
}

// MMA issuer of k_fwd_main (one thread).  A function of its own so its few
// live values stay in registers whatever the other roles need.
__device__ __noinline__ void fwd_mma_role(FwdBars& bars, uint32_t tmem, uint32_t sbase,
                                          const int4* tasks, const TaskWalk walk,
                                          volatile int* abort_flag) {
  const int64_t my_n = walk.n;
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
  bool ok = true;
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
    return true;
  };
  int cur_kv = task_rec(tasks, 0, walk).w;
  int next_kv = task_rec(tasks, 1, walk).w;
  ok = wait_kv() && issue_S(0);
  for (int64_t it = 0; ok && it < my_n; ++it) {
    const int st = int(it & 1);
    const int next2_kv = task_rec(tasks, it + 2, walk).w;
    const bool same = (it + 1 < my_n) && next_kv == cur_kv;
    if (same && !issue_S(it + 1)) break;
    if (!wait(bars.p_full[st], uint32_t((it >> 1) & 1))) break;
    // one O_part stage: the epilogue must have read O_part(it-1)
    if (it >= 1 && !wait(bars.o_free, uint32_t((it - 1) & 1))) break;
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

__global__ void __launch_bounds__(kFwdThreads, 1)
    k_fwd_main(const __grid_constant__ FwdParams prm, const __grid_constant__ CUtensorMap mapQ,
               const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
               const __grid_constant__ CUtensorMap mapPool) {
  grid_dep_wait();
  grid_dep_release();
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
  const int64_t ntasks = skip_sh ? 0 : p.header[kHdrFTasks];
  const TaskWalk walk = task_walk<kFwdChunk>(ntasks);
  const int64_t my_n = walk.n;
  const int4* tasks = reinterpret_cast<const int4*>(p.ftasks);

  if (warp == 0) {
    // ---------------- TMA producer (records and tokens prefetched one task ahead)
    if (lane == 0 && my_n > 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      int prev_kv = -1;
      int64_t kv_loads = 0, it = 0;
      int4 rec = task_rec(tasks, 0, walk), rec1 = task_rec(tasks, 1, walk);
      int32_t tok[kTaskQueries];
      {
        const TaskView tv = decode_task(rec);
#pragma unroll
        for (int qi = 0; qi < kTaskQueries; ++qi) tok[qi] = task_token(p.col, tv, qi);
      }
      for (; it < my_n; ++it) {
        const TaskView tv = decode_task(rec);
        const int4 rec2 = task_rec(tasks, it + 2, walk);
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
          load_kv_tiles(sbase + kSmK, sbase + kSmV, &mapK, &mapV, b, tv.g, tv.key_start);
          ++kv_loads;
          prev_kv = tv.sub;
        }
        const int st = int(it & 1);
        if (it >= 2 &&
            !mbar_wait(smem_u32(&bars.q_empty[st]), uint32_t(((it >> 1) - 1) & 1), abort_flag))
          break;
#ifdef MSA_TEST_STARVE
        if (!(g_starve_fwd == 2 && blockIdx.x == 0 && it == 0))
#endif
        {
          const uint32_t b = smem_u32(&bars.q_full[st]);
          mbar_arrive_expect_tx(b, kTileBytes);
          load_q_tile(sbase + kSmQ + st * kTileBytes, &mapQ, b, tok, tv.g);
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
    if (lane == 0 && my_n > 0) fwd_mma_role(bars, tmem, sbase, tasks, walk, abort_flag);
  } else if (warp < 10) {
    // ---------------- softmax (warps 2-5: even tasks, 6-9: odd tasks)
    const int quad = warp & 3;
    const int par = (warp - 2) >> 2;
    const int row = quad * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    const int qi = row >> 4, hh = row & 15;
    // A row takes part when its query is real and not grouped (grouped
    // queries are the group kernel's): jmax = last visible key, -1 if not.
    auto row_jmax = [&](const TaskView& tv, int32_t tok) {
      return (qi < tv.nq && !p.grouped[int64_t(tv.g) * p.T + tok])
                 ? min(tok - tv.key_start, tv.key_len - 1)
                 : -1;
    };
    // Row data of this warpgroup's next task (it+2) is loaded while task it
    // runs, in two steps so no load result is consumed right after it is
    // issued: the row's token at the top of task it, its shift M and
    // grouped flag after the exponentials.
    int4 rec1 = task_rec(tasks, par + 2, walk);
    int jmax_c = -1;
    float m2_c = 0.f;
    if (par < my_n) {
      const TaskView tv = decode_task(task_rec(tasks, par, walk));
      const int32_t tok = task_token(p.col, tv, qi);
      jmax_c = row_jmax(tv, tok);
      m2_c = prm.M2[int64_t(tok) * kQHeads + tv.g * kHeadsPerGroup + hh];
    }
    for (int64_t it = par; it < my_n; it += 2) {
      const int st = int(it & 1);
      const int jmax = jmax_c;
      const float m2 = m2_c;
      const int4 rec2 = task_rec(tasks, it + 4, walk);
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
        jmax_c = row_jmax(tn, ntok);
        m2_c = prm.M2[int64_t(ntok) * kQHeads + tn.g * kHeadsPerGroup + hh];
      }
      // the epilogue of task it-2 has read this stage's row scalars
      if (it >= 2 &&
          !mbar_wait_warp(smem_u32(&bars.rs_free[st]), uint32_t(((it >> 1) - 1) & 1), abort_flag))
        break;
      s_alpha[st][row] = jmax >= 0 ? fast_exp2(mxc - m2) : 0.f;
      s_lrow[st][row] = jmax >= 0 ? lsum : -1.f;  // -1: the row takes no part
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
    // pool with four bulk tensor reductions per query.
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    const int qi = row >> 4, hh = row & 15;
    const uint32_t stage_q = sbase + kSmStage + uint32_t(qi) * 8192u;
    const uint32_t stage_row = stage_q + uint32_t(hh) * 128u;
    const uint32_t swz = uint32_t(hh & 7);
    if (lane == 0 && my_n > 0) tma_prefetch_desc(&mapPool);
    int4 rec = task_rec(tasks, 0, walk), rec1 = task_rec(tasks, 1, walk);
    // the row's token is loaded one task ahead
    int32_t tok_c = my_n > 0 ? task_token(p.col, decode_task(rec), qi) : 0;
    for (int64_t it = 0; it < my_n; ++it) {
      const int st = int(it & 1);
      const TaskView tv = decode_task(rec);
      const int4 rec2 = task_rec(tasks, it + 2, walk);
      const int32_t tok = tok_c;
      tok_c = task_token(p.col, decode_task(rec1), qi);  // rec1: a valid record
      const int64_t grow = int64_t(tok) * kQHeads + tv.g * kHeadsPerGroup + hh;
      if (!mbar_wait_warp(smem_u32(&bars.o_full), uint32_t(it & 1), abort_flag)) break;
      // p_full(it) completed before o_full(it); waiting on it makes the
      // softmax's row scalars visible here.
      if (!mbar_wait_warp(smem_u32(&bars.p_full[st]), uint32_t((it >> 1) & 1), abort_flag)) break;
      tc_fence_after();
      const float alpha = s_alpha[st][row];
      const float lrow = s_lrow[st][row];
      mbar_arrive(smem_u32(&bars.rs_free[st]));
      const float mul = alpha * prm.vscale[tv.g];
      // the warp's two queries take part? (rows 0 and 16 of the warp)
      const bool take0 = __shfl_sync(0xffffffffu, lrow, 0) >= 0.f;
      const bool take1 = __shfl_sync(0xffffffffu, lrow, 16) >= 0.f;
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
          if (j ? take1 : take0) {
            const int y = (j ? tok_hi : tok) * kQHeads + tv.g * kHeadsPerGroup;
#pragma unroll
            for (int cq = cq0; cq < cq0 + 2; ++cq)
              tma_reduce_add_2d(&mapPool, sbase + kSmStage + uint32_t(qj) * 8192u + cq * 2048u,
                                cq * 32, y);
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
      stage_box(0, v0);
      stage_box(1, v1);
      tmem_ld32(obase + 64, v0);
      tmem_ld32(obase + 96, v1);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) issue_pair(0);
      __syncwarp();
      tmem_ld_wait();
      reg_fence32(v0);
      reg_fence32(v1);
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.o_free));  // O_part read: the next P.V may overwrite it
      if (lane == 0) bulk_wait_read1();  // previous task's boxes 2-3 read
      __syncwarp();
      stage_box(2, v0);
      stage_box(3, v1);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) issue_pair(2);
      if (lrow > 0.f) atomicAdd(prm.lsum + grow, alpha * lrow);
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

// ------------------------------------------------------------ fwd_group
// One item: octet A (and octet B) of one index head, whose tokens all see the
// same blocks (uniform item), or which lie in a query block b small enough to
// walk all of blocks 0 .. b with each token's rows masked to the blocks it
// selected (dense item).  The CTA walks those blocks: per block S_A = Q_A K^T and
// S_B = Q_B K^T, P = exp(s - m_ref) as fp16 over S's own first 64 columns,
// then O_A += P_A V and O_B += P_B V, O accumulating in TMEM across the
// blocks.  m_ref is a row's reference maximum, set from the first block the
// row takes part in and raised only when a later block's maximum passes it by more than
// 15 octaves (so P < 2^16 stays in fp16); then O and the row sum are
// rescaled in place.  After the last block the softmax warps write their
// octet's O = acc / l and LSE: no pool, no finalize, no shift bound.
//
// P overwrites S, so the next S of an octet comes after its P.V; tensor-core
// operations of one issuing thread run in issue order, so that needs no
// wait.  The issue order S_A(j), P_B(j-1).V, S_B(j), P_A(j).V leaves each
// octet's softmax two groups of MMAs (~1000 cycles) to run in.
// Warp roles (320 threads):
//   0     TMA producer: Q tiles of octets A and B (one buffer each: the next
//         item's tile of an octet loads once the octet's last S of the
//         current item is done), K and V per block (two stages each)
//   1     MMA issuer (TMEM owner)
//   2-5   softmax and epilogue of octet A (thread = tile row = TMEM lane)
//   6-9   the same for octet B
// TMEM: S_A [0,128) with P_A over [0,64), S_B [128,256) with P_B over
// [128,192), O_A [256,384), O_B [384,512).
// Items are placed by decreasing cost; CTA c takes items c, 2G-1-c, 2G+c, ...
// (a snake over the G CTAs) so that the CTAs' totals balance.
constexpr int kGrpThreads = 320;
constexpr uint32_t kGsQ = 0, kGsK = 65536, kGsV = 131072;
constexpr uint32_t kGrpSmem = kGsV + 2 * kTileBytes + 1024;
constexpr uint32_t kGtO = 256;
constexpr float kRaiseOctaves = 15.f;  // P = 2^(s - m_ref) < 2^16 fits fp16

struct GrpBars {
  uint64_t q_full[2], q_empty[2], k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2],
      p_full[2], o_full[2], o_free[2], fin;
};

__device__ __forceinline__ int64_t item_index(int64_t i) {
  const int64_t c = (i & 1) ? int64_t(gridDim.x) - 1 - blockIdx.x : int64_t(blockIdx.x);
  return i * gridDim.x + c;
}
__device__ __forceinline__ int64_t item_count(int64_t n) {
  const int64_t full = n / gridDim.x, rem = n % gridDim.x;
  const int64_t c = (full & 1) ? int64_t(gridDim.x) - 1 - blockIdx.x : int64_t(blockIdx.x);
  return full + (c < rem ? 1 : 0);
}

// P = 2^(s c2 - mref) of one tile row (TMEM columns [cs, cs + 128) of the
// thread's lane) as fp16 pairs into pk (pair k = columns 2k, 2k+1), keys
// after jmax masked when MASK; S is left intact.  Returns the sum of the
// fp32 values; *tmax gets the row's maximum raw score.
template <bool MASK>
__device__ __forceinline__ float row_exp_regs(uint32_t cs, int jmax, float c2, float mref,
                                              uint32_t (&pk)[64], float* tmax) {
  const uint64_t cc = f2_pack(__float_as_uint(c2), __float_as_uint(c2));
  const uint64_t nm = f2_pack(__float_as_uint(-mref), __float_as_uint(-mref));
  uint64_t ls[2] = {0ull, 0ull};
  float m0 = -INFINITY, m1 = -INFINITY;
  auto expo = [&](const uint32_t (&r)[16], int l, int c) {
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      float x0 = __uint_as_float(r[j]), x1 = __uint_as_float(r[j + 1]);
      const uint64_t x2 = f2_fma(f2_pack(r[j], r[j + 1]), cc, nm);
      float p0 = fast_exp2(f2_lo(x2)), p1 = fast_exp2(f2_hi(x2));
      if (MASK) {
        p0 = j <= l ? p0 : 0.f;
        p1 = j + 1 <= l ? p1 : 0.f;
        x0 = j <= l ? x0 : -INFINITY;
        x1 = j + 1 <= l ? x1 : -INFINITY;
      }
      if (j & 2) m1 = fmax3(m1, x0, x1); else m0 = fmax3(m0, x0, x1);
      ls[(j >> 1) & 1] =
          f2_add(ls[(j >> 1) & 1], f2_pack(__float_as_uint(p0), __float_as_uint(p1)));
      pk[8 * c + (j >> 1)] = pack_f16x2(p0, p1);
    }
  };
  // chunk c+1 loads while chunk c is exponentiated
  uint32_t r0[16], r1[16];
  tmem_ld16(cs, r0);
  tmem_ld_wait();
  reg_fence16(r0);
#pragma unroll
  for (int c = 0; c < 8; c += 2) {
    tmem_ld16(cs + 16 * c + 16, r1);
    expo(r0, jmax - 16 * c, c);
    tmem_ld_wait();
    reg_fence16(r1);
    if (c < 6) tmem_ld16(cs + 16 * c + 32, r0);
    expo(r1, jmax - 16 * c - 16, c + 1);
    if (c < 6) {
      tmem_ld_wait();
      reg_fence16(r0);
    }
  }
  *tmax = fmaxf(m0, m1);
  const uint64_t s2 = f2_add(ls[0], ls[1]);
  return f2_lo(s2) + f2_hi(s2);
}

// MMA issuer of k_fwd_group (one thread).
__device__ __noinline__ void grp_mma_role(GrpBars& bars, uint32_t tmem, uint32_t sbase,
                                          const int32_t* items, int64_t my_n,
                                          volatile int* abort_flag) {
  constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);  // Q . K^T  (bf16)
  constexpr uint32_t idPV = idesc_f16_f32(128, 128, 0, 1);  // P . V    (fp16, P in TMEM)
  auto wait = [&](uint64_t& bar, uint32_t ph) {
    return mbar_wait(smem_u32(&bar), ph, abort_flag);
  };
  const uint64_t kQ0 = sdesc_sw128(sbase + kGsQ, 16u, 1024u);
  const uint64_t kK0 = sdesc_sw128(sbase + kGsK, 16u, 1024u);
  const uint64_t mV0 = sdesc_sw128(sbase + kGsV, 16384u, 1024u);
  constexpr uint64_t kStage = kTileBytes >> 4;
  auto kstep = [](int kk) { return uint64_t((kk >> 2) * 1024 + (kk & 3) * 2); };
  auto mstep = [](int kk) { return uint64_t(kk) * 128u; };
  int64_t nblk = 0;          // blocks walked (K / V stage phases)
  int64_t nx[2] = {0, 0};    // blocks per octet slot (s_full / p_full phases)
  int64_t ix[2] = {0, 0};    // items per octet slot (o_full / o_free phases)
  int64_t qu[2] = {0, 0};    // uses of the two Q buffers
  auto issue_S = [&](int x, int stg) {
    const uint64_t bq = kQ0 + uint64_t(x) * kStage;
    const uint64_t bk = kK0 + uint64_t(stg) * kStage;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ss(tmem + 128 * x, bq + kstep(kk), bk + kstep(kk), idS, kk > 0);
    umma_commit(smem_u32(&bars.s_full[x]));
  };
  // O_x += P_x . V of the block in V stage stg (first block: O_x = ...)
  auto issue_PV = [&](int x, int stg, bool first) -> bool {
    if (!wait(bars.p_full[x], uint32_t(nx[x] & 1))) return false;
    if (first && ix[x] > 0 && !wait(bars.o_free[x], uint32_t((ix[x] - 1) & 1))) return false;
    tc_fence_after();
    const uint64_t bv = mV0 + uint64_t(stg) * kStage;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ts(tmem + kGtO + 128 * x, tmem + 128 * x + kk * 8, bv + mstep(kk), idPV,
              (!first || kk > 0) ? 1u : 0u);
    ++nx[x];
    return true;
  };
  // the previous block's P_B . V, issued after the next S_A
  bool pend = false, pend_first = false, pend_last = false;
  int pend_stg = 0;
  auto flush_B = [&]() -> bool {
    if (!pend) return true;
    if (!issue_PV(1, pend_stg, pend_first)) return false;
    umma_commit(smem_u32(&bars.v_empty[pend_stg]));
    if (pend_last) {
      umma_commit(smem_u32(&bars.o_full[1]));
      ++ix[1];
    }
    pend = false;
    return true;
  };
  bool ok = true;
  for (int64_t i = 0; ok && i < my_n; ++i) {
    const ItemView iv = decode_item(items + item_index(i) * kItemWords);
    const bool hasB = iv.tokB >= 0;
    for (int j = 0; j < iv.nsel; ++j) {
      const int stg = int(nblk & 1);
      const uint32_t ph = uint32_t((nblk >> 1) & 1);
      const bool last = j + 1 == iv.nsel;
      if (!wait(bars.k_full[stg], ph)) { ok = false; break; }
      if (j == 0 && !wait(bars.q_full[0], uint32_t(qu[0] & 1))) { ok = false; break; }
      tc_fence_after();
      issue_S(0, stg);
      if (last) {
        umma_commit(smem_u32(&bars.q_empty[0]));
        ++qu[0];
      }
      if (!flush_B()) { ok = false; break; }
      if (hasB) {
        if (j == 0 && !wait(bars.q_full[1], uint32_t(qu[1] & 1))) { ok = false; break; }
        tc_fence_after();
        issue_S(1, stg);
        if (last) {
          umma_commit(smem_u32(&bars.q_empty[1]));
          ++qu[1];
        }
      }
      umma_commit(smem_u32(&bars.k_empty[stg]));  // K of this block: both S issued
      if (!wait(bars.v_full[stg], ph)) { ok = false; break; }
      if (!issue_PV(0, stg, j == 0)) { ok = false; break; }
      if (last) {
        umma_commit(smem_u32(&bars.o_full[0]));
        ++ix[0];
      }
      if (hasB) {
        pend = true;
        pend_stg = stg;
        pend_first = j == 0;
        pend_last = last;
      } else {
        umma_commit(smem_u32(&bars.v_empty[stg]));
      }
      ++nblk;
    }
  }
  if (ok) flush_B();
  umma_commit(smem_u32(&bars.fin));
  mbar_wait_drain(smem_u32(&bars.fin), 0);
}

__global__ void __launch_bounds__(kGrpThreads, 1)
    k_fwd_group(const __grid_constant__ FwdParams prm, const __grid_constant__ CUtensorMap mapQ,
                const __grid_constant__ CUtensorMap mapK,
                const __grid_constant__ CUtensorMap mapV) {
  grid_dep_wait();
  grid_dep_release();
  extern __shared__ uint8_t smem_raw[];
  __shared__ GrpBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, skip_sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const msa_plan& p = prm.plan;
  volatile int* abort_flag = &abort_sh;

  if (threadIdx.x == 0) {
    abort_sh = 0;
    skip_sh = plan_failed(p.header) ? 1 : 0;
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.q_full[i]), 1);
      mbar_init(smem_u32(&bars.q_empty[i]), 1);
      mbar_init(smem_u32(&bars.k_full[i]), 1);
      mbar_init(smem_u32(&bars.k_empty[i]), 1);
      mbar_init(smem_u32(&bars.v_full[i]), 1);
      mbar_init(smem_u32(&bars.v_empty[i]), 1);
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.p_full[i]), 128);
      mbar_init(smem_u32(&bars.o_full[i]), 1);
      mbar_init(smem_u32(&bars.o_free[i]), 128);
    }
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
  const int64_t nitems = skip_sh ? 0 : p.header[kHdrItems];
  const int64_t my_n = item_count(nitems);
  const int32_t* items = p.items;
  const DocInfo* dinfo = reinterpret_cast<const DocInfo*>(p.doc_info);

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0 && my_n > 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      int64_t nblk = 0, qu[2] = {0, 0};
      bool ok = true;
      auto load_q = [&](int buf, int32_t tok0, int nq, int g) -> bool {
        if (qu[buf] > 0 &&
            !mbar_wait(smem_u32(&bars.q_empty[buf]), uint32_t((qu[buf] - 1) & 1), abort_flag))
          return false;
#ifdef MSA_TEST_STARVE
        if (g_starve_fwd == 1 && blockIdx.x == 0 && buf == 0 && qu[0] == 0) {
          ++qu[buf];
          return true;
        }
#endif
        int32_t tok[kTaskQueries];
#pragma unroll
        for (int qi = 0; qi < kTaskQueries; ++qi) tok[qi] = tok0 + (qi < nq ? qi : nq - 1);
        const uint32_t b = smem_u32(&bars.q_full[buf]);
        mbar_arrive_expect_tx(b, kTileBytes);
        load_q_tile(sbase + kGsQ + buf * kTileBytes, &mapQ, b, tok, g);
        ++qu[buf];
        return true;
      };
      // K and V of one block into stage nblk & 1 of their rings
      auto load_kv = [&](int g, int32_t key_start) -> bool {
        const int stg = int(nblk & 1);
        const uint32_t ph = uint32_t(((nblk >> 1) - 1) & 1);
        if (nblk >= 2 && !mbar_wait(smem_u32(&bars.k_empty[stg]), ph, abort_flag)) return false;
        uint32_t b = smem_u32(&bars.k_full[stg]);
        mbar_arrive_expect_tx(b, kTileBytes);
        tma_load_3d(sbase + kGsK + stg * kTileBytes, &mapK, b, 0, g, key_start);
        tma_load_3d(sbase + kGsK + stg * kTileBytes + 16384, &mapK, b, 64, g, key_start);
        if (nblk >= 2 && !mbar_wait(smem_u32(&bars.v_empty[stg]), ph, abort_flag)) return false;
        b = smem_u32(&bars.v_full[stg]);
        mbar_arrive_expect_tx(b, kTileBytes);
        tma_load_3d(sbase + kGsV + stg * kTileBytes, &mapV, b, 0, g, key_start);
        tma_load_3d(sbase + kGsV + stg * kTileBytes + 16384, &mapV, b, 64, g, key_start);
        ++nblk;
        return true;
      };
      for (int64_t i = 0; ok && i < my_n; ++i) {
        const int32_t* it = items + item_index(i) * kItemWords;
        const ItemView iv = decode_item(it);
        const int32_t dstart = dinfo[iv.doc].start;
        if (i + 1 < my_n) {
          // the next item's Q tiles into L2: their loads then wait on L2,
          // not on HBM, between this item's last S and the next item's first
          const ItemView nv = decode_item(items + item_index(i + 1) * kItemWords);
          for (int x = 0; x < (nv.tokB >= 0 ? 2 : 1); ++x) {
            const int32_t t0 = x ? nv.tokB : nv.tokA;
            const int nq = x ? nv.nqB : nv.nqA;
            for (int qi = 0; qi < nq; ++qi) {
              const int y = (t0 + qi) * kQHeads + nv.g * kHeadsPerGroup;
              tma_prefetch_l2_2d(&mapQ, 0, y);
              tma_prefetch_l2_2d(&mapQ, 64, y);
            }
          }
        }
        // A's tile, K/V of the first block, B's tile, the other blocks
        ok = load_q(0, iv.tokA, iv.nqA, iv.g);
        for (int j = 0; ok && j < iv.nsel; ++j) {
          ok = load_kv(iv.g, dstart + (iv.dense ? j : it[4 + j]) * kBlock);
          if (ok && j == 0 && iv.tokB >= 0) ok = load_q(1, iv.tokB, iv.nqB, iv.g);
        }
      }
      if (*abort_flag) {  // let armed copies land before the CTA exits
        for (int64_t j = (nblk >= 2 ? nblk - 2 : 0); j < nblk; ++j) {
          mbar_wait_drain(smem_u32(&bars.k_full[j & 1]), uint32_t((j >> 1) & 1));
          mbar_wait_drain(smem_u32(&bars.v_full[j & 1]), uint32_t((j >> 1) & 1));
        }
        for (int b = 0; b < 2; ++b)
          if (qu[b] > 0) mbar_wait_drain(smem_u32(&bars.q_full[b]), uint32_t((qu[b] - 1) & 1));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0 && my_n > 0) grp_mma_role(bars, tmem, sbase, items, my_n, abort_flag);
  } else {
    // ---------------- softmax + epilogue of octet x (warps 2-5: A, 6-9: B)
    const int x = (warp - 2) >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    const int qi = row >> 4, hh = row & 15;
    const uint32_t cs = tmem + lane_base + 128 * x;
    const uint32_t co = tmem + lane_base + kGtO + 128 * x;
    int64_t nx = 0, ix = 0;
    for (int64_t i = 0; i < my_n; ++i) {
      const int32_t* it = items + item_index(i) * kItemWords;
      const ItemView iv = decode_item(it);
      if (x == 1 && iv.tokB < 0) continue;
      const int32_t tok0 = x ? iv.tokB : iv.tokA;
      const int nq = x ? iv.nqB : iv.nqA;
      const int32_t tok = tok0 + (qi < nq ? qi : nq - 1);
      const int32_t dstart = dinfo[iv.doc].start;
      // dense item: the row's token takes part in block j where bit j is set
      const int tw = 4 + 2 * (8 * x + qi);
      const uint64_t tmask =
          iv.dense ? (uint64_t(uint32_t(it[tw])) | uint64_t(uint32_t(it[tw + 1])) << 32) : ~0ull;
      float mref = -INFINITY, lsum = 0.f;
      bool ok = true;
      for (int j = 0; j < iv.nsel; ++j) {
        const int32_t key_start = dstart + (iv.dense ? j : it[4 + j]) * kBlock;
        const int jmax = qi < nq && ((tmask >> j) & 1ull) ? min(tok - key_start, kBlock - 1) : -1;
        // S_x(j) complete: so is P_x(j-1) . V, which was issued before it
        if (!mbar_wait_warp(smem_u32(&bars.s_full[x]), uint32_t(nx & 1), abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // Without masks when every row of the warp sees the whole block or
        // none of it (a dense item's token that did not select the block):
        // such rows are computed unmasked and then zeroed.
        const bool full = __all_sync(0xffffffffu, jmax == kBlock - 1 || jmax < 0);
        if (j == 0) {  // the item's first block sets the reference
          const float mx = full ? tile_row_max<false>(cs, jmax) : tile_row_max<true>(cs, jmax);
          mref = jmax >= 0 ? mx * prm.c2 : -INFINITY;
        }
        uint32_t pk[64];
        float tmax;
        auto row_exp = [&]() {
          if (!full) return row_exp_regs<true>(cs, jmax, prm.c2, mref, pk, &tmax);
          float l = row_exp_regs<false>(cs, jmax, prm.c2, mref, pk, &tmax);
          if (jmax < 0) {
#pragma unroll
            for (int k = 0; k < 64; ++k) pk[k] = 0u;
            l = 0.f;
            tmax = -INFINITY;
          }
          return l;
        };
        float ls = row_exp();
        const float mxc = tmax * prm.c2;
        const bool raise = j > 0 && jmax >= 0 && mxc > mref + kRaiseOctaves;
        if (__any_sync(0xffffffffu, raise)) {
          // rescale O (complete up to block j-1) and the row sum by
          // 2^(mref - mxc), then redo the exponentials (S is still intact)
          const float f = raise ? fast_exp2(mref - mxc) : 1.f;
          lsum *= f;
          if (raise) mref = mxc;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(co + 32 * c, o);
            tmem_ld_wait();
            reg_fence32(o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32_nc(co + 32 * c, o);
          }
          ls = row_exp();
        }
        lsum += ls;
        // P over the first 64 columns of S (all of S has been read)
        tmem_st32_nc(cs, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
        tmem_st32_nc(cs + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.p_full[x]));
        ++nx;
      }
      if (!ok) break;
      // ---- epilogue: O = acc / l, LSE
      if (!mbar_wait_warp(smem_u32(&bars.o_full[x]), uint32_t(ix & 1), abort_flag)) break;
      ++ix;
      tc_fence_after();
      uint32_t o[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(co + 32 * c, o[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < 4; ++c) reg_fence32(o[c]);
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.o_free[x]));  // the next item's P.V may overwrite O_x
      if (qi < nq) {
        const int64_t grow = int64_t(tok) * kQHeads + iv.g * kHeadsPerGroup + hh;
        if (!(lsum > 0.f) || !isfinite(lsum)) {
          const int32_t k = atomicAdd(prm.list, 1);  // the fallback writes this row
          prm.list[1 + k] = int32_t(grow);
        } else {
          const float inv = prm.vscale[iv.g] / lsum;
          uint4* dst = reinterpret_cast<uint4*>(prm.O + grow * kHeadDim);
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t* v = &o[c][8 * u];
              dst[4 * c + u] = make_uint4(
                  pack_bf16x2(__uint_as_float(v[0]) * inv, __uint_as_float(v[1]) * inv),
                  pack_bf16x2(__uint_as_float(v[2]) * inv, __uint_as_float(v[3]) * inv),
                  pack_bf16x2(__uint_as_float(v[4]) * inv, __uint_as_float(v[5]) * inv),
                  pack_bf16x2(__uint_as_float(v[6]) * inv, __uint_as_float(v[7]) * inv));
            }
          prm.lse[grow] = (mref + __log2f(lsum)) * kLn2;
        }
      }
    }
  }

  // ---------------- teardown
  if (threadIdx.x == 0 && abort_sh) raise_status(p.header, MSA_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ fwd_finalize
// Pooled rows (the plan's list): O = pool / sum -> bf16 and LSE =
// (M + log2 sum) ln 2.  Each warp finishes eight rows per step (16 lanes x 8
// elements per row; the eight rows are heads of one token and index head),
// all loads issued before any use.  Grouped rows were written by the group
// kernel.  Rows whose sum
// underflowed are listed for the fallback.
constexpr int kFinRowsPerWarp = 8;
__global__ void __launch_bounds__(256) k_fwd_finalize(msa_plan p, const float* M2,
                                                      const float* lsum, const float* pool,
                                                      __nv_bfloat16* O, float* lse,
                                                      int32_t* list) {
  grid_dep_wait();
  grid_dep_release();
  if (plan_failed(p.header)) return;
  const int lane = threadIdx.x & 31, sub = lane & 15;
  // the plan's list of pooled rows: entry 4 t + g is the 16 rows of token t,
  // index head g, finished by a warp in two steps of eight
  const int64_t nsteps = 2 * p.header[kHdrRows];
  const int64_t nwarps = int64_t(gridDim.x) * blockDim.x / 32;
  for (int64_t j = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) / 32; j < nsteps;
       j += nwarps) {
    const int32_t ent = p.rows[j >> 1];
    const int64_t r0 = (int64_t(ent >> 2) * kQHeads + (ent & 3) * kHeadsPerGroup) +
                       (j & 1) * kFinRowsPerWarp;
    float4 a[4], b[4];
    float m2[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = r0 + 2 * i + (lane >> 4);
      const float4* src = reinterpret_cast<const float4*>(pool + row * kHeadDim) + 2 * sub;
      a[i] = src[0];
      b[i] = src[1];
      m2[i] = M2[row];
      l[i] = lsum[row];
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = r0 + 2 * i + (lane >> 4);
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
        out = make_uint4(pack_bf16x2(a[i].x * inv, a[i].y * inv), pack_bf16x2(a[i].z * inv, a[i].w * inv),
                         pack_bf16x2(b[i].x * inv, b[i].y * inv), pack_bf16x2(b[i].z * inv, b[i].w * inv));
        L = (m2[i] + __log2f(l[i])) * kLn2;
      }
      reinterpret_cast<uint4*>(O + row * kHeadDim)[sub] = out;
      if (sub == 0) lse[row] = L;
    }
    // the eight rows' pool lines are dead (the fallback does not read the
    // pool): drop them from L2, a lane per 128-byte line
    __syncwarp();
    if ((sub & 3) == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        l2_discard_line(pool + (r0 + 2 * i + (lane >> 4)) * kHeadDim + 8 * sub);
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
  grid_dep_wait();
  grid_dep_release();
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
int device_sm_count();                                                       // msa_api.cu

size_t forward_workspace_bytes(const msa_plan& p) { return fwd_layout(p).total; }

cudaError_t launch_forward(const msa_plan& p, const void* q, const void* k, const void* v,
                           float scale, void* o, float* lse, void* ws, cudaStream_t s) {
  const FwdLayout L = fwd_layout(p);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* M2 = reinterpret_cast<float*>(w + L.off_m);
  float* lsum = reinterpret_cast<float*>(w + L.off_l);
  float* vmax = reinterpret_cast<float*>(w + L.off_vmax);
  float* pool = reinterpret_cast<float*>(w + L.off_pool);
  float* kmax = reinterpret_cast<float*>(w + L.off_kmax);
  int32_t* list = reinterpret_cast<int32_t*>(w + L.off_list);
  uint4* v16 = reinterpret_cast<uint4*>(w + L.off_v16);
  float* vscale = reinterpret_cast<float*>(w + L.off_vscale);
  const float c2 = scale * kLog2e;

  // V tiles are read from the fp16 copy (same element size, same map shape)
  CUtensorMap mQ, mK, mV, mPool;
  if (make_map_rows(&mQ, q, p.T * kQHeads) != CUDA_SUCCESS ||
      make_map_kv(&mK, k, p.T) != CUDA_SUCCESS || make_map_kv(&mV, v16, p.T) != CUDA_SUCCESS ||
      make_map_pool32(&mPool, pool, p.T * kQHeads) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(q);
  const __nv_bfloat16* kb = static_cast<const __nv_bfloat16*>(k);
  const __nv_bfloat16* vb = static_cast<const __nv_bfloat16*>(v);
  __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
  cudaError_t e;
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(k_fwd_main, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_fwd_group, cudaFuncAttributeMaxDynamicSharedMemorySize, kGrpSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  FwdParams prm{p, M2, kmax, vmax, pool, lsum, list, ob, lse, vscale, c2};
  const unsigned grid = unsigned(device_sm_count());
  // Every kernel may start during its predecessor's tail (launch_k) and
  // waits for it before touching memory; a caller's kernel that never
  // signals counts as signalling when it completes.
  launch_begin("fwd_kmax", s);
  e = launch_k(true, k_fwd_kmax, dim3(unsigned(p.nb_cap)), dim3(kKmaxThreads), 0, s, p, kb, vb,
               kmax, vmax, list, v16);
  launch_end("fwd_kmax", s);
  if (e != cudaSuccess) return e;
  launch_begin("fwd_v16", s);
  e = launch_k(true, k_fwd_v16, dim3(grid * 4), dim3(256), 0, s, p, vb, (const float*)vmax, v16,
               vscale);
  launch_end("fwd_v16", s);
  if (e != cudaSuccess) return e;
  // The group kernel needs neither the row shifts nor the pool: it runs
  // first, on the K / V / Q lines the earlier kernels left in L2.
  launch_begin("fwd_group", s);
  e = launch_k(true, k_fwd_group, dim3(grid), dim3(kGrpThreads), kGrpSmem, s, prm, mQ, mK, mV);
  launch_end("fwd_group", s);
  if (e != cudaSuccess) return e;
  launch_begin("fwd_rows", s);
  e = launch_k(true, k_fwd_rows, dim3(grid * 16), dim3(256), 0, s, p, qb,
               (const float*)kmax, (const float*)vmax, c2, M2, lsum, pool);
  launch_end("fwd_rows", s);
  if (e != cudaSuccess) return e;
  launch_begin("fwd_main", s);
  e = launch_k(true, k_fwd_main, dim3(grid), dim3(kFwdThreads), kFwdSmem, s, prm, mQ, mK, mV,
               mPool);
  launch_end("fwd_main", s);
  if (e != cudaSuccess) return e;
  launch_begin("fwd_finalize", s);
  e = launch_k(true, k_fwd_finalize, dim3(grid * 16), dim3(256), 0, s, p, (const float*)M2,
               (const float*)lsum, (const float*)pool, ob, lse, list);
  launch_end("fwd_finalize", s);
  if (e != cudaSuccess) return e;
  launch_begin("fwd_fallback", s);
  e = launch_k(true, k_fwd_fallback, dim3(grid * 4), dim3(256), 0, s, p, qb, kb, vb, c2,
               (const int32_t*)list, ob, lse);
  launch_end("fwd_fallback", s);
  return e;
}

}  // namespace msa
