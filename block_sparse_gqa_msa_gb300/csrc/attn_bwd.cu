// attn_bwd.cu - MSA backward: dQ [T,64,128], dK, dV [T,4,128].
//
// Launch sequence as on the pages (NeMo-Automodel PR "feat(minimax-m3) ...",
// "Custom backward design"): delta preprocess -> zero gradient pools -> main
// attention backward -> BF16 gradient finalization.  The main kernel is
// KV-parallel like the pages' design (API page msa_backward_sm100): each CTA
// walks task rows, keeps the bucket's K/V block resident in shared memory,
// loads the task's 8 query rows of Q and dO per tile, and per tile issues five
// 128x128x128 tcgen05 contractions with fp32 accumulators in tensor memory:
//   S  = Q K^T,   dP = dO V^T,                       (TMEM cols 0 and 128)
//   dV += P^T dO, dK += dS^T Q  over the bucket run,   (TMEM cols 256, 384)
//   dQ  = dS K                                         (TMEM cols 0, after S)
// with P = exp(S * scale - LSE) and dS = P (dP - delta).  dV / dK are flushed
// with fp32 L2 reductions when the run of tasks on the same block ends; dQ is
// reduced per tile into an fp32 pool.  The finalize casts the pools to bf16.
//
// Kernels, in launch order:
//   bwd_delta     delta = rowsum(dO * O); zero the dQ / dK / dV pools
//   bwd_main      the tensor-core tile loop
//   bwd_finalize  pools -> bf16 dQ, dK, dV
#include "common.cuh"
#include "sm100.cuh"

namespace msa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct BwdLayout {
  size_t off_delta, off_dq, off_dk, off_dv, total;
};
BwdLayout bwd_layout(const msa_plan& p) {
  BwdLayout L{};
  const int64_t rows = p.T * kQHeads;
  size_t o = 0;
  L.off_delta = o; o = align_up(o + sizeof(float) * rows, 256);
  L.off_dq = o;    o = align_up(o + sizeof(float) * rows * kHeadDim, 256);
  L.off_dk = o;    o = align_up(o + sizeof(float) * p.T * kKVHeads * kHeadDim, 256);
  L.off_dv = o;    o = align_up(o + sizeof(float) * p.T * kKVHeads * kHeadDim, 256);
  L.total = o;
  return L;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ------------------------------------------------------------ bwd_delta
// One warp per row (t, h): delta = sum_c dO * O (bf16 inputs, fp32 sum), and
// zero the row of the dQ pool; rows < 4T also zero one row of dK and dV pools.
__global__ void __launch_bounds__(256) k_bwd_delta(msa_plan p, const __nv_bfloat16* O,
                                                   const __nv_bfloat16* dO, float* delta,
                                                   float* dq_pool, float* dk_pool,
                                                   float* dv_pool) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (row >= p.T * kQHeads || plan_failed(p.header)) return;
  const uint2 a = reinterpret_cast<const uint2*>(O + row * kHeadDim)[lane];
  const uint2 b = reinterpret_cast<const uint2*>(dO + row * kHeadDim)[lane];
  float s = bf16_lo(a.x) * bf16_lo(b.x);
  s = fmaf(bf16_hi(a.x), bf16_hi(b.x), s);
  s = fmaf(bf16_lo(a.y), bf16_lo(b.y), s);
  s = fmaf(bf16_hi(a.y), bf16_hi(b.y), s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) delta[row] = s;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  reinterpret_cast<float4*>(dq_pool + row * kHeadDim)[lane] = zero;
  if (row < p.T * kKVHeads) {
    reinterpret_cast<float4*>(dk_pool + row * kHeadDim)[lane] = zero;
    reinterpret_cast<float4*>(dv_pool + row * kHeadDim)[lane] = zero;
  }
}

// ------------------------------------------------------------ bwd_main
constexpr int kBwdThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 compute / reduce
constexpr uint32_t kTileBytes = 32768;
constexpr uint32_t kSmK = 0, kSmV = 32768, kSmQ = 65536, kSmDO = 98304, kSmP = 131072,
                   kSmDS = 163840, kSmStage = 196608;
constexpr uint32_t kStageFloats = 32 * 33;
constexpr uint32_t kBwdSmem = kSmStage + 4 * kStageFloats * 4 + 1024;

constexpr uint32_t kTmS = 0, kTmDP = 128, kTmDV = 256, kTmDK = 384, kTmDQ = 0;

struct BwdBars {
  uint64_t kv_full, kv_empty, qdo_full, qdo_empty, sdp_full, pds_full, dq_full, dq_free, dkv_free,
      fin;
};

struct BwdParams {
  msa_plan plan;
  const float* lse;
  const float* delta;
  float* dq_pool;
  float* dk_pool;
  float* dv_pool;
  float c2;     // scale * log2(e)
  float scale;
  int chunk;
};

__device__ __forceinline__ int64_t cta_task(int64_t i, int chunk) {
  return (int64_t(blockIdx.x) + (i / chunk) * gridDim.x) * chunk + (i % chunk);
}
__device__ __forceinline__ int64_t cta_task_count(int64_t ntasks, int chunk) {
  const int64_t nchunks = (ntasks + chunk - 1) / chunk;
  if (int64_t(blockIdx.x) >= nchunks) return 0;
  const int64_t mine = (nchunks - 1 - blockIdx.x) / gridDim.x + 1;
  const int64_t last_chunk = blockIdx.x + (mine - 1) * gridDim.x;
  return (mine - 1) * chunk + (ntasks - last_chunk * chunk < chunk ? ntasks - last_chunk * chunk
                                                                    : chunk);
}

// Reduce 32 rows x 32 fp32 columns held one row per lane (r[]) into global
// rows dst (one pointer per lane, already offset to the column chunk) with
// coalesced 16-byte L2 reductions: the warp transposes through `stage`.
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
      const float* s = stage + src * 33 + c4;
      red_add_v4_f32(d + c4, s[0], s[1], s[2], s[3]);
    }
  }
  __syncwarp();
}

__global__ void __launch_bounds__(kBwdThreads, 1)
    k_bwd_main(const __grid_constant__ BwdParams prm, const __grid_constant__ CUtensorMap mapQ,
               const __grid_constant__ CUtensorMap mapDO, const __grid_constant__ CUtensorMap mapK,
               const __grid_constant__ CUtensorMap mapV) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdBars bars;
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
    mbar_init(smem_u32(&bars.qdo_full), 1);
    mbar_init(smem_u32(&bars.qdo_empty), 1);
    mbar_init(smem_u32(&bars.sdp_full), 1);
    mbar_init(smem_u32(&bars.pds_full), 128);
    mbar_init(smem_u32(&bars.dq_full), 1);
    mbar_init(smem_u32(&bars.dq_free), 128);
    mbar_init(smem_u32(&bars.dkv_free), 128);
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
      tma_prefetch_desc(&mapDO);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      int prev_sub = -1;
      int64_t kv_loads = 0, it = 0;
      for (; it < my_n; ++it) {
        const TaskView tv = decode_task(tasks[cta_task(it, prm.chunk)]);
        if (tv.sub != prev_sub) {
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
          prev_sub = tv.sub;
        }
        if (it >= 1 && !mbar_wait(smem_u32(&bars.qdo_empty), uint32_t((it - 1) & 1), abort_flag))
          break;
        const uint32_t b = smem_u32(&bars.qdo_full);
        mbar_arrive_expect_tx(b, 2 * kTileBytes);
        for (int qi = 0; qi < kTaskQueries; ++qi) {
          const int32_t tok = p.col[tv.col_begin + (qi < tv.nq ? qi : tv.nq - 1)];
          const int y = tok * kQHeads + tv.g * kHeadsPerGroup;
          tma_load_2d(sbase + kSmQ + qi * 2048, &mapQ, b, 0, y);
          tma_load_2d(sbase + kSmQ + 16384 + qi * 2048, &mapQ, b, 64, y);
          tma_load_2d(sbase + kSmDO + qi * 2048, &mapDO, b, 0, y);
          tma_load_2d(sbase + kSmDO + 16384 + qi * 2048, &mapDO, b, 64, y);
        }
      }
      if (*abort_flag) {  // let armed copies land before the CTA exits
        if (kv_loads > 0) mbar_wait_drain(smem_u32(&bars.kv_full), uint32_t((kv_loads - 1) & 1));
        if (it > 0) mbar_wait_drain(smem_u32(&bars.qdo_full), uint32_t((it - 1) & 1));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0 && my_n > 0) {
      constexpr uint32_t idKK = idesc_bf16_f32(128, 128, 0, 0);  // S, dP
      constexpr uint32_t idMM = idesc_bf16_f32(128, 128, 1, 1);  // dV, dK
      constexpr uint32_t idKM = idesc_bf16_f32(128, 128, 0, 1);  // dQ
      int cur_sub = -1;
      int64_t kv_loads = 0, seg_done = 0;
      bool first_in_seg = true;
      for (int64_t it = 0; it < my_n; ++it) {
        const TaskView tv = decode_task(tasks[cta_task(it, prm.chunk)]);
        if (tv.sub != cur_sub) {
          if (it > 0) umma_commit(smem_u32(&bars.kv_empty));
          if (!mbar_wait(smem_u32(&bars.kv_full), uint32_t(kv_loads & 1), abort_flag)) break;
          ++kv_loads;
          cur_sub = tv.sub;
          first_in_seg = true;
        }
        if (!mbar_wait(smem_u32(&bars.qdo_full), uint32_t(it & 1), abort_flag)) break;
        if (it >= 1 && !mbar_wait(smem_u32(&bars.dq_free), uint32_t((it - 1) & 1), abort_flag))
          break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + kTmS, desc_kmajor(sbase + kSmQ, kk), desc_kmajor(sbase + kSmK, kk), idKK,
                  kk > 0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + kTmDP, desc_kmajor(sbase + kSmDO, kk), desc_kmajor(sbase + kSmV, kk),
                  idKK, kk > 0);
        umma_commit(smem_u32(&bars.sdp_full));
        if (!mbar_wait(smem_u32(&bars.pds_full), uint32_t(it & 1), abort_flag)) break;
        if (first_in_seg && seg_done > 0 &&
            !mbar_wait(smem_u32(&bars.dkv_free), uint32_t((seg_done - 1) & 1), abort_flag))
          break;
        tc_fence_after();
        const uint32_t acc0 = first_in_seg ? 0u : 1u;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + kTmDV, desc_mnmajor(sbase + kSmP, kk), desc_mnmajor(sbase + kSmDO, kk),
                  idMM, kk > 0 ? 1u : acc0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + kTmDK, desc_mnmajor(sbase + kSmDS, kk), desc_mnmajor(sbase + kSmQ, kk),
                  idMM, kk > 0 ? 1u : acc0);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_ss(tmem + kTmDQ, desc_kmajor(sbase + kSmDS, kk), desc_mnmajor(sbase + kSmK, kk),
                  idKM, kk > 0);
        umma_commit(smem_u32(&bars.dq_full));
        umma_commit(smem_u32(&bars.qdo_empty));
        first_in_seg = false;
        const bool seg_end =
            (it + 1 == my_n) || decode_task(tasks[cta_task(it + 1, prm.chunk)]).sub != cur_sub;
        if (seg_end) ++seg_done;
      }
      umma_commit(smem_u32(&bars.fin));
      mbar_wait_drain(smem_u32(&bars.fin), 0);
    }
  } else {
    // ---------------- compute: softmax / dS, dQ reduction, dK / dV flush
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    float* stage = reinterpret_cast<float*>(smem + kSmStage) + (warp - 2) * kStageFloats;
    for (int64_t it = 0; it < my_n; ++it) {
      const TaskView tv = decode_task(tasks[cta_task(it, prm.chunk)]);
      const int qi = row >> 4, hh = row & 15;
      const bool row_valid = qi < tv.nq;
      const int32_t tok = p.col[tv.col_begin + (row_valid ? qi : tv.nq - 1)];
      const int64_t grow = int64_t(tok) * kQHeads + tv.g * kHeadsPerGroup + hh;
      int jmax = tok - tv.key_start;
      if (jmax > tv.key_len - 1) jmax = tv.key_len - 1;
      if (!row_valid) jmax = -1;
      const float lse2 = prm.lse[grow] * kLog2e;
      const float dl = prm.delta[grow];
      if (!mbar_wait_warp(smem_u32(&bars.sdp_full), uint32_t(it & 1), abort_flag)) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t s[32], dp[32];
        tmem_ld32(tmem + lane_base + kTmS + c * 32, s);
        tmem_ld32(tmem + lane_base + kTmDP + c * 32, dp);
        tmem_ld_wait();
        uint32_t pp[16], pd[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int k0 = c * 32 + j;
          const float p0 = (k0 <= jmax) ? fast_exp2(fmaf(__uint_as_float(s[j]), prm.c2, -lse2)) : 0.f;
          const float p1 =
              (k0 + 1 <= jmax) ? fast_exp2(fmaf(__uint_as_float(s[j + 1]), prm.c2, -lse2)) : 0.f;
          const float d0 = p0 * (__uint_as_float(dp[j]) - dl);
          const float d1 = p1 * (__uint_as_float(dp[j + 1]) - dl);
          pp[j >> 1] = pack_bf16x2(p0, p1);
          pd[j >> 1] = pack_bf16x2(d0, d1);
        }
        const uint32_t off = (c >> 1) * 16384 + row * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint32_t ch = (((c & 1) * 4 + u) ^ (row & 7)) * 16;
          st_shared_v4(sbase + kSmP + off + ch, pp[4 * u], pp[4 * u + 1], pp[4 * u + 2], pp[4 * u + 3]);
          st_shared_v4(sbase + kSmDS + off + ch, pd[4 * u], pd[4 * u + 1], pd[4 * u + 2], pd[4 * u + 3]);
        }
      }
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars.pds_full));

      // dQ: reduce scale * (dS K) rows into the pool
      if (!mbar_wait_warp(smem_u32(&bars.dq_full), uint32_t(it & 1), abort_flag)) break;
      tc_fence_after();
      float* dq_row = prm.dq_pool + grow * kHeadDim;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + lane_base + kTmDQ + c * 32, r);
        tmem_ld_wait();
        warp_reduce_rows(stage, r, prm.scale, dq_row + c * 32, row_valid);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.dq_free));

      // end of a run of tasks on this K/V block: flush dV and dK (lane = key)
      const bool seg_end =
          (it + 1 == my_n) || decode_task(tasks[cta_task(it + 1, prm.chunk)]).sub != tv.sub;
      if (seg_end) {
        const bool key_valid = row < tv.key_len;
        const int64_t krow = (int64_t(tv.key_start) + row) * kKVHeads + tv.g;
        float* dv_row = prm.dv_pool + krow * kHeadDim;
        float* dk_row = prm.dk_pool + krow * kHeadDim;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_base + kTmDV + c * 32, r);
          tmem_ld_wait();
          warp_reduce_rows(stage, r, 1.f, dv_row + c * 32, key_valid);
          tmem_ld32(tmem + lane_base + kTmDK + c * 32, r);
          tmem_ld_wait();
          warp_reduce_rows(stage, r, prm.scale, dk_row + c * 32, key_valid);
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.dkv_free));
      }
    }
  }

  if (threadIdx.x == 0 && abort_sh) raise_status(p.header, MSA_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ bwd_finalize
// fp32 pools -> bf16 outputs; one warp per 128-element row.
__global__ void __launch_bounds__(256) k_bwd_finalize(msa_plan p, const float* dq_pool,
                                                      const float* dk_pool, const float* dv_pool,
                                                      __nv_bfloat16* dq, __nv_bfloat16* dk,
                                                      __nv_bfloat16* dv) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nq = p.T * kQHeads, nk = p.T * kKVHeads;
  if (row >= nq + 2 * nk || plan_failed(p.header)) return;
  const float* src;
  __nv_bfloat16* dst;
  if (row < nq) {
    src = dq_pool + row * kHeadDim;
    dst = dq + row * kHeadDim;
  } else if (row < nq + nk) {
    src = dk_pool + (row - nq) * kHeadDim;
    dst = dk + (row - nq) * kHeadDim;
  } else {
    src = dv_pool + (row - nq - nk) * kHeadDim;
    dst = dv + (row - nq - nk) * kHeadDim;
  }
  const float4 x = reinterpret_cast<const float4*>(src)[lane];
  reinterpret_cast<uint2*>(dst)[lane] = make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
}

}  // namespace

CUresult make_map_rows(CUtensorMap* m, const void* base, int64_t rows);
CUresult make_map_kv(CUtensorMap* m, const void* base, int64_t T);
int device_sm_count();

size_t backward_workspace_bytes(const msa_plan& p) { return bwd_layout(p).total; }

cudaError_t launch_backward(const msa_plan& p, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout, float scale,
                            void* dq, void* dk, void* dv, void* ws, cudaStream_t s) {
  const BwdLayout L = bwd_layout(p);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* delta = reinterpret_cast<float*>(w + L.off_delta);
  float* dq_pool = reinterpret_cast<float*>(w + L.off_dq);
  float* dk_pool = reinterpret_cast<float*>(w + L.off_dk);
  float* dv_pool = reinterpret_cast<float*>(w + L.off_dv);

  CUtensorMap mQ, mDO, mK, mV;
  if (make_map_rows(&mQ, q, p.T * kQHeads) != CUDA_SUCCESS ||
      make_map_rows(&mDO, dout, p.T * kQHeads) != CUDA_SUCCESS ||
      make_map_kv(&mK, k, p.T) != CUDA_SUCCESS || make_map_kv(&mV, v, p.T) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  const int64_t rows = p.T * kQHeads;
  launch_begin("bwd_delta", s);
  k_bwd_delta<<<unsigned((rows + 7) / 8), 256, 0, s>>>(
      p, static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), delta,
      dq_pool, dk_pool, dv_pool);
  launch_end("bwd_delta", s);

  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(k_bwd_main, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  BwdParams prm{p, lse, delta, dq_pool, dk_pool, dv_pool, scale * kLog2e, scale, 8};
  launch_begin("bwd_main", s);
  k_bwd_main<<<unsigned(device_sm_count()), kBwdThreads, kBwdSmem, s>>>(prm, mQ, mDO, mK, mV);
  launch_end("bwd_main", s);
  const int64_t frows = rows + 2 * p.T * kKVHeads;
  launch_begin("bwd_finalize", s);
  k_bwd_finalize<<<unsigned((frows + 7) / 8), 256, 0, s>>>(
      p, dq_pool, dk_pool, dv_pool, static_cast<__nv_bfloat16*>(dq),
      static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv));
  launch_end("bwd_finalize", s);
  return cudaGetLastError();
}

}  // namespace msa
