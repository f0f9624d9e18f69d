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
// without a second pass over the scores: every task exponentiates against
// the same per-row shift M[t,h] = scale * |q_th| * max_{selected v} max_{j in v}
// |k_jg| (log2 units), which bounds every score of the row (Cauchy-Schwarz),
// and adds its unnormalised P.V and row sum into fp32 pools with L2
// reductions.  The finalize divides.  Rows whose sum underflows (the bound far
// above the true maximum) are recomputed exactly by a fallback kernel.
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
struct FwdLayout {
  size_t off_m, off_l, off_l2, off_pool, off_kmax, off_vmax, off_list, total;
};
FwdLayout fwd_layout(const msa_plan& p) {
  FwdLayout L{};
  const int64_t rows = p.T * kQHeads;
  size_t o = 0;
  L.off_m = o;    o = align_up(o + sizeof(float) * rows, 256);
  L.off_l = o;    o = align_up(o + sizeof(float) * rows, 256);
  L.off_l2 = o;   o = align_up(o + sizeof(float) * rows, 256);
  L.off_pool = o; o = align_up(o + sizeof(float) * rows * kHeadDim, 256);
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
// One warp per (token, index head): M2 = c2 * |q_th| * kmax_sel for the 16
// heads (-inf when the row sees no key), and zero the row's pool and sum.
__global__ void __launch_bounds__(256) k_fwd_rows(msa_plan p, const __nv_bfloat16* Q,
                                                  const float* kmax, float c2, float* M2,
                                                  float* lsum, float* lsum2, float* pool) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (wid >= p.T * kKVHeads || plan_failed(p.header)) return;
  const int64_t t = wid >> 2;
  const int g = int(wid & 3);
  const int d = doc_of_token(p.doc_offsets, p.num_docs, t);
  const DocInfo di = reinterpret_cast<const DocInfo*>(p.doc_info)[d];
  const int64_t qb = (t - di.start) / kBlock;
  float km = -1.f;
  if (lane < kTopK) {
    const int32_t v = p.q2k[(int64_t(g) * p.T + t) * kTopK + lane];
    if (v >= 0 && v <= qb) km = kmax[int64_t(g) * p.nb_cap + di.blk_base + v];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) km = fmaxf(km, __shfl_xor_sync(0xffffffffu, km, o));
  // 16 heads x 128 dims = 4 KB of Q: lanes 0-15 take head 2i, 16-31 head 2i+1.
  const __nv_bfloat16* qrow = Q + (t * kQHeads + g * kHeadsPerGroup) * kHeadDim;
  float* prow = pool + (t * kQHeads + g * kHeadsPerGroup) * kHeadDim;
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
      M2[row] = km < 0.f ? -INFINITY : c2 * sqrtf(s) * km;
      lsum[row] = 0.f;
      lsum2[row] = 0.f;
    }
  }
  float4* z = reinterpret_cast<float4*>(prow);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
  for (int i = lane; i < kHeadsPerGroup * kHeadDim / 4; i += 32) z[i] = zero;
}

// ------------------------------------------------------------ fwd_main
// Warp roles: 0 TMA producer, 1 MMA issuer (and TMEM owner), 2-5 softmax +
// epilogue (thread = tile row = TMEM lane), 6 converts each V tile to fp16.
// TMEM: S in columns [0,128) / [128,256) (two stages), O_part in
// [256,384) / [384,512).
//
// Per task the softmax works relative to the tile's own row maximum m
// (P = exp(s - m) in (0, 1], fp16), and the epilogue rescales the partial
// P.V and row sums by exp(m - M) before adding them to the pools, so every
// task of a row lands on the same shift M.
constexpr int kFwdThreads = 224;
constexpr uint32_t kTileBytes = 32768;
constexpr uint32_t kSmK = 0, kSmV = 32768, kSmQ = 65536, kSmP = 131072, kSmStage = 163840;
constexpr uint32_t kStageFloats = 32 * 33;
constexpr uint32_t kFwdSmem = kSmStage + 4 * kStageFloats * 4 + 1024;

struct FwdBars {
  uint64_t kv_full, kv_empty, v_ready, q_full[2], q_empty[2], s_full[2], s_free[2], p_full,
      p_free, o_full[2], o_free[2], fin;
};

struct FwdParams {
  msa_plan plan;
  const float* M2;
  const float* vmax;
  float* pool;
  float* lsum;   // sum of the fp32 weights (gives LSE)
  float* lsum2;  // sum of the fp16-rounded weights (normalises O)
  float c2;
  int chunk;
};

// Task i of the CTA's walk: chunks of `chunk` consecutive tasks go round-robin
// over the CTAs, so all CTAs advance through the task list together.
__device__ __forceinline__ int64_t cta_task(int64_t i, int chunk) {
  return (int64_t(blockIdx.x) + (i / chunk) * gridDim.x) * chunk + (i % chunk);
}
__device__ __forceinline__ int64_t cta_task_count(int64_t ntasks, int chunk) {
  const int64_t nchunks = (ntasks + chunk - 1) / chunk;
  if (int64_t(blockIdx.x) >= nchunks) return 0;
  const int64_t mine = (nchunks - 1 - blockIdx.x) / gridDim.x + 1;  // chunks of this CTA
  const int64_t last_chunk = blockIdx.x + (mine - 1) * gridDim.x;
  return (mine - 1) * chunk + (ntasks - last_chunk * chunk < chunk ? ntasks - last_chunk * chunk
                                                                    : chunk);
}

// Reduce 32 rows x 32 fp32 columns held one row per lane into global rows
// (one destination pointer per lane, already offset to the column chunk)
// with coalesced 16-byte L2 reductions; the warp transposes through `stage`.
__device__ __forceinline__ void warp_reduce_rows(float* stage, const uint32_t (&r)[32], float mul,
                                                 float* dst, bool valid) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 32; ++j) stage[lane * 33 + j] = __uint_as_float(r[j]) * mul;
  __syncwarp();
#pragma unroll
  for (int rr = 0; rr < 32; rr += 4) {
    const int src = rr + (lane >> 3);
    const int c4 = (lane & 7) * 4;
    float* d = reinterpret_cast<float*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dst), src));
    const bool v = __shfl_sync(0xffffffffu, valid ? 1 : 0, src) != 0;
    if (v) {
      const float* sp = stage + src * 33 + c4;
      red_add_v4_f32(d + c4, sp[0], sp[1], sp[2], sp[3]);
    }
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kFwdThreads, 1)
    k_fwd_main(const __grid_constant__ FwdParams prm, const __grid_constant__ CUtensorMap mapQ,
               const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdBars bars;
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
    mbar_init(smem_u32(&bars.kv_full), 1);
    mbar_init(smem_u32(&bars.kv_empty), 1);
    mbar_init(smem_u32(&bars.v_ready), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.q_full[i]), 1);
      mbar_init(smem_u32(&bars.q_empty[i]), 1);
      mbar_init(smem_u32(&bars.s_full[i]), 1);
      mbar_init(smem_u32(&bars.s_free[i]), 128);
      mbar_init(smem_u32(&bars.o_full[i]), 1);
      mbar_init(smem_u32(&bars.o_free[i]), 128);
    }
    mbar_init(smem_u32(&bars.p_full), 128);
    mbar_init(smem_u32(&bars.p_free), 1);
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
  const int64_t my_n = cta_task_count(ntasks, prm.chunk);
  const int4* tasks = reinterpret_cast<const int4*>(p.tasks);

  if (warp == 0) {
    // ---------------- TMA producer
    if (lane == 0 && my_n > 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      int prev_kv = -1;
      int64_t kv_loads = 0, it = 0;
      for (; it < my_n; ++it) {
        const TaskView tv = decode_task(tasks[cta_task(it, prm.chunk)]);
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
        for (int qi = 0; qi < kTaskQueries; ++qi) {
          const int32_t tok = p.col[tv.col_begin + (qi < tv.nq ? qi : tv.nq - 1)];
          const int y = tok * kQHeads + tv.g * kHeadsPerGroup;
          tma_load_2d(dst + qi * 2048, &mapQ, b, 0, y);
          tma_load_2d(dst + 16384 + qi * 2048, &mapQ, b, 64, y);
        }
      }
      if (*abort_flag) {  // let armed copies land before the CTA exits
        if (kv_loads > 0) mbar_wait_drain(smem_u32(&bars.kv_full), uint32_t((kv_loads - 1) & 1));
        for (int64_t j = (it >= 2 ? it - 2 : 0); j < it; ++j)
          mbar_wait_drain(smem_u32(&bars.q_full[j & 1]), uint32_t((j >> 1) & 1));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0 && my_n > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, 0, 0);  // Q . K^T   (bf16)
      constexpr uint32_t idPV = idesc_f16_f32(128, 128, 0, 1);  // P . V     (fp16, V MN-major)
      int64_t kv_loads = 0;
      bool ok = true, need_v = false;
      auto issue_S = [&](int64_t it) -> bool {
        const int st = int(it & 1);
        if (!mbar_wait(smem_u32(&bars.q_full[st]), uint32_t((it >> 1) & 1), abort_flag))
          return false;
        if (it >= 2 &&
            !mbar_wait(smem_u32(&bars.s_free[st]), uint32_t(((it >> 1) - 1) & 1), abort_flag))
          return false;
        tc_fence_after();
        const uint32_t sq = sbase + kSmQ + st * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + st * 128, desc_kmajor(sq, kk), desc_kmajor(sbase + kSmK, kk), idS,
                  kk > 0);
        umma_commit(smem_u32(&bars.s_full[st]));
        umma_commit(smem_u32(&bars.q_empty[st]));
        return true;
      };
      auto wait_kv = [&]() -> bool {
        if (!mbar_wait(smem_u32(&bars.kv_full), uint32_t(kv_loads & 1), abort_flag)) return false;
        ++kv_loads;
        need_v = true;
        return true;
      };
      int cur_kv = decode_task(tasks[cta_task(0, prm.chunk)]).sub;
      ok = wait_kv() && issue_S(0);
      for (int64_t it = 0; ok && it < my_n; ++it) {
        const int st = int(it & 1);
        int next_kv = -1;
        if (it + 1 < my_n) next_kv = decode_task(tasks[cta_task(it + 1, prm.chunk)]).sub;
        const bool same = (it + 1 < my_n) && next_kv == cur_kv;
        if (same && !issue_S(it + 1)) { ok = false; break; }
        if (!mbar_wait(smem_u32(&bars.p_full), uint32_t(it & 1), abort_flag)) { ok = false; break; }
        if (it >= 2 &&
            !mbar_wait(smem_u32(&bars.o_free[st]), uint32_t(((it >> 1) - 1) & 1), abort_flag)) {
          ok = false;
          break;
        }
        if (need_v) {
          if (!mbar_wait(smem_u32(&bars.v_ready), uint32_t((kv_loads - 1) & 1), abort_flag)) {
            ok = false;
            break;
          }
          need_v = false;
        }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + 256 + st * 128, desc_kmajor(sbase + kSmP, kk),
                  desc_mnmajor(sbase + kSmV, kk), idPV, kk > 0);
        umma_commit(smem_u32(&bars.o_full[st]));
        umma_commit(smem_u32(&bars.p_free));
        if (it + 1 < my_n && !same) {
          umma_commit(smem_u32(&bars.kv_empty));
          cur_kv = next_kv;
          if (!wait_kv() || !issue_S(it + 1)) { ok = false; break; }
        }
      }
      // Make sure no MMA is still running before TMEM is released.
      umma_commit(smem_u32(&bars.fin));
      mbar_wait_drain(smem_u32(&bars.fin), 0);
    }
  } else if (warp == 6) {
    // ---------------- V tile bf16 -> fp16 (scaled by an exact power of two)
    if (my_n > 0) {
      int prev_kv = -1;
      int64_t kv_loads = 0;
      for (int64_t it = 0; it < my_n; ++it) {
        const TaskView tv = decode_task(tasks[cta_task(it, prm.chunk)]);
        if (tv.sub == prev_kv) continue;
        prev_kv = tv.sub;
        if (!mbar_wait_warp(smem_u32(&bars.kv_full), uint32_t(kv_loads & 1), abort_flag)) break;
        ++kv_loads;
        const float sc = v_scale_in(prm.vmax[tv.sub]);
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
  } else {
    // ---------------- softmax + epilogue (warps 2-5)
    const int quad = warp & 3;            // TMEM lane quadrant of this warp
    const int row = quad * 32 + lane;     // tile row = TMEM lane
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    float* stage = reinterpret_cast<float*>(smem + kSmStage) + (warp - 2) * kStageFloats;
    for (int64_t it = 0; it < my_n; ++it) {
      const int st = int(it & 1);
      const TaskView tv = decode_task(tasks[cta_task(it, prm.chunk)]);
      const int qi = row >> 4, hh = row & 15;
      const bool row_valid = qi < tv.nq;
      const int32_t tok = p.col[tv.col_begin + (row_valid ? qi : tv.nq - 1)];
      const int64_t grow = int64_t(tok) * kQHeads + tv.g * kHeadsPerGroup + hh;
      int jmax = tok - tv.key_start;
      if (jmax > tv.key_len - 1) jmax = tv.key_len - 1;
      if (!row_valid) jmax = -1;
      const float m2 = prm.M2[grow];
      const float vs = v_scale_in(prm.vmax[tv.sub]);
      if (!mbar_wait_warp(smem_u32(&bars.s_full[st]), uint32_t((it >> 1) & 1), abort_flag)) break;
      tc_fence_after();
      // pass 1: the tile row's maximum over visible keys (raw scores)
      float mx = -INFINITY;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + st * 128 + c * 32, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (c * 32 + j <= jmax) mx = fmaxf(mx, __uint_as_float(r[j]));
      }
      const float mxc = (jmax >= 0) ? mx * prm.c2 : 0.f;
      if (it >= 1 && !mbar_wait_warp(smem_u32(&bars.p_free), uint32_t((it - 1) & 1), abort_flag))
        break;
      // pass 2: P = exp(s - m) as fp16 into the P tile; exact and rounded sums
      float l_exact = 0.f, l_round = 0.f;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + st * 128 + c * 32, r);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int k0 = c * 32 + j;
          const float x0 = (k0 <= jmax) ? fast_exp2(fmaf(__uint_as_float(r[j]), prm.c2, -mxc)) : 0.f;
          const float x1 =
              (k0 + 1 <= jmax) ? fast_exp2(fmaf(__uint_as_float(r[j + 1]), prm.c2, -mxc)) : 0.f;
          const uint32_t w2 = pack_f16x2(x0, x1);
          l_exact += x0 + x1;
          l_round += f16_lo(w2) + f16_hi(w2);
          pk[j >> 1] = w2;
        }
        const uint32_t prow = sbase + kSmP + (c >> 1) * 16384 + row * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t chunk = ((c & 1) * 4 + u) ^ (row & 7);
          st_shared_v4(prow + chunk * 16, pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.s_free[st]));
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars.p_full));

      // epilogue: pool[row] += exp(m - M) * O_partial / vscale
      const float alpha = row_valid ? fast_exp2(mxc - m2) : 0.f;
      if (!mbar_wait_warp(smem_u32(&bars.o_full[st]), uint32_t((it >> 1) & 1), abort_flag)) break;
      tc_fence_after();
      float* dst_row = prm.pool + grow * kHeadDim;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + 256 + st * 128 + c * 32, r);
        tmem_ld_wait();
        warp_reduce_rows(stage, r, alpha / vs, dst_row + c * 32, row_valid);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.o_free[st]));
      if (row_valid) {
        atomicAdd(prm.lsum + grow, alpha * l_exact);
        atomicAdd(prm.lsum2 + grow, alpha * l_round);
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
// One warp per row (t, h).
__global__ void __launch_bounds__(256) k_fwd_finalize(msa_plan p, const float* M2,
                                                      const float* lsum, const float* lsum2,
                                                      const float* pool, __nv_bfloat16* O,
                                                      float* lse, int32_t* list) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (row >= p.T * kQHeads) return;
  if (plan_failed(p.header)) return;
  const float m2 = M2[row];
  const float l = lsum[row];
  uint2 out = make_uint2(0u, 0u);
  bool write = true;
  float L = -INFINITY;
  if (m2 != -INFINITY) {
    if (!(l >= kUnderflowSum) || !isfinite(l)) {
      write = false;  // the fallback kernel writes this row
      if (lane == 0) {
        const int32_t k = atomicAdd(list, 1);
        list[1 + k] = int32_t(row);
      }
    } else {
      const float4 x = reinterpret_cast<const float4*>(pool + row * kHeadDim)[lane];
      const float inv = 1.f / lsum2[row];
      out.x = pack_bf16x2(x.x * inv, x.y * inv);
      out.y = pack_bf16x2(x.z * inv, x.w * inv);
      L = (m2 + __log2f(l)) * kLn2;
    }
  }
  if (write) {
    reinterpret_cast<uint2*>(O + row * kHeadDim)[lane] = out;
    if (lane == 0) lse[row] = L;
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
int device_sm_count();                                                       // msa_api.cu

size_t forward_workspace_bytes(const msa_plan& p) { return fwd_layout(p).total; }

cudaError_t launch_forward(const msa_plan& p, const void* q, const void* k, const void* v,
                           float scale, void* o, float* lse, void* ws, cudaStream_t s) {
  const FwdLayout L = fwd_layout(p);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* M2 = reinterpret_cast<float*>(w + L.off_m);
  float* lsum = reinterpret_cast<float*>(w + L.off_l);
  float* lsum2 = reinterpret_cast<float*>(w + L.off_l2);
  float* vmax = reinterpret_cast<float*>(w + L.off_vmax);
  float* pool = reinterpret_cast<float*>(w + L.off_pool);
  float* kmax = reinterpret_cast<float*>(w + L.off_kmax);
  int32_t* list = reinterpret_cast<int32_t*>(w + L.off_list);
  const float c2 = scale * kLog2e;

  CUtensorMap mQ, mK, mV;
  if (make_map_rows(&mQ, q, p.T * kQHeads) != CUDA_SUCCESS ||
      make_map_kv(&mK, k, p.T) != CUDA_SUCCESS || make_map_kv(&mV, v, p.T) != CUDA_SUCCESS)
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
      p, static_cast<const __nv_bfloat16*>(q), kmax, c2, M2, lsum, lsum2, pool);
  launch_end("fwd_rows", s);

  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(k_fwd_main, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  FwdParams prm{p, M2, vmax, pool, lsum, lsum2, c2, 8};
  launch_begin("fwd_main", s);
  k_fwd_main<<<unsigned(device_sm_count()), kFwdThreads, kFwdSmem, s>>>(prm, mQ, mK, mV);
  launch_end("fwd_main", s);
  const int64_t rows = p.T * kQHeads;
  launch_begin("fwd_finalize", s);
  k_fwd_finalize<<<unsigned((rows + 7) / 8), 256, 0, s>>>(
      p, M2, lsum, lsum2, pool, static_cast<__nv_bfloat16*>(o), lse, list);
  launch_end("fwd_finalize", s);
  launch_begin("fwd_fallback", s);
  k_fwd_fallback<<<unsigned(device_sm_count() * 4), 256, 0, s>>>(
      p, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), c2, list, static_cast<__nv_bfloat16*>(o), lse);
  launch_end("fwd_fallback", s);
  return cudaGetLastError();
}

}  // namespace msa
