// attn_bwd.cu - MSA backward: dQ [T,64,128], dK, dV [T,4,128].
//
// Launch sequence as on the pages (NeMo-Automodel PR "feat(minimax-m3) ...",
// "Custom backward design"): delta preprocess -> zero gradient pools -> main
// attention backward -> gradient finalization.  The main kernel is KV-parallel
// and, like the pages' design (API page msa_backward_sm100), issues its five
// tcgen05 GEMMs transposed so that the key block is the MMA's M dimension:
//   S^T  = K Q^T,   dP^T = V dO^T                 (TMEM cols [0,128), [128,256))
//   P^T  = exp(S^T * scale - LSE),  dS^T = P^T (dP^T - delta)
//   dV  += P^T dO,  dK += dS^T Q   (A operands read from TMEM; cols 256, 384)
//   dQ^T = K^T dS^T                 (dS from shared memory; cols [128,256))
// TMEM lane = key for S/dP/dV/dK, so the per-key softmax work is one thread
// per key; lane = head dimension for dQ^T, so one warp reduces 32 consecutive
// dQ elements of a row at a time (coalesced).  dV / dK accumulate over a run
// of tasks that share the K/V block and are flushed with fp32 L2 reductions;
// dQ is reduced per tile into an fp16 (default), bf16 or fp32 pool.
//
// bwd_main runs 14 warps: a TMA producer, an MMA issuer, eight compute warps
// (P^T, dS^T; two per TMEM lane quadrant, each owning 64 q-rows) and four
// reduce warps (dQ^T staging + bulk tensor reduction, dV / dK flush).
//
// Kernels, in launch order:
//   bwd_delta     delta = rowsum(dO * O); zero the dQ / dK / dV pools
//   bwd_main      the tensor-core tile loop
//   bwd_finalize  pools -> bf16 dQ, dK, dV
#include "common.cuh"
#include "sm100.cuh"

#include <cstring>

namespace msa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

struct BwdLayout {
  size_t off_delta, off_dq, off_dk, off_dv, total;
};
size_t dq_elem_bytes(const msa_plan& p) { return p.dq_accum == MSA_DQ_ACCUM_F32 ? 4 : 2; }
BwdLayout bwd_layout(const msa_plan& p) {
  BwdLayout L{};
  const int64_t rows = p.T * kQHeads;
  size_t o = 0;
  L.off_delta = o; o = align_up(o + sizeof(float) * rows, 256);
  L.off_dq = o;    o = align_up(o + dq_elem_bytes(p) * rows * kHeadDim, 256);
  L.off_dk = o;    o = align_up(o + sizeof(float) * p.T * kKVHeads * kHeadDim, 256);
  L.off_dv = o;    o = align_up(o + sizeof(float) * p.T * kKVHeads * kHeadDim, 256);
  L.total = o;
  return L;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ------------------------------------------------------------ bwd_delta
// One thread per 8 elements: delta[row] = sum_c dO * O over the row's 128
// elements (16 threads per row), plus zeroing of the pools.  Each thread
// handles 4 rows' worth of work so several loads are in flight.
constexpr int kDeltaRowsPerWarp = 8;
__global__ void __launch_bounds__(256) k_bwd_delta(msa_plan p, const __nv_bfloat16* O,
                                                   const __nv_bfloat16* dO, float* delta,
                                                   uint4* dq_pool, int64_t dq_pool_vec,
                                                   float4* dkv_pool, int64_t dkv_vec) {
  if (plan_failed(p.header)) return;
  const int lane = threadIdx.x & 31;
  const int64_t rows = p.T * kQHeads;
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t r0 = warp0 * kDeltaRowsPerWarp;
  // lanes 0-15 -> row r, lanes 16-31 -> row r+1 (8 elements each)
  uint4 a[kDeltaRowsPerWarp / 2], b[kDeltaRowsPerWarp / 2];
#pragma unroll
  for (int i = 0; i < kDeltaRowsPerWarp / 2; ++i) {
    const int64_t row = r0 + 2 * i + (lane >> 4);
    if (row < rows) {
      a[i] = reinterpret_cast<const uint4*>(O + row * kHeadDim)[lane & 15];
      b[i] = reinterpret_cast<const uint4*>(dO + row * kHeadDim)[lane & 15];
    } else {
      a[i] = b[i] = make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int i = 0; i < kDeltaRowsPerWarp / 2; ++i) {
    const uint32_t x[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
    const uint32_t y[4] = {b[i].x, b[i].y, b[i].z, b[i].w};
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s = fmaf(bf16_lo(x[e]), bf16_lo(y[e]), s);
      s = fmaf(bf16_hi(x[e]), bf16_hi(y[e]), s);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const int64_t row = r0 + 2 * i + (lane >> 4);
    if ((lane & 15) == 0 && row < rows) delta[row] = s;
  }
  // zero the pools with a grid-stride loop of 16-byte stores
  const int64_t nthreads = int64_t(gridDim.x) * blockDim.x;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int64_t i = tid; i < dq_pool_vec; i += nthreads) dq_pool[i] = z;
  const float4 zf = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = tid; i < dkv_vec; i += nthreads) dkv_pool[i] = zf;
}

// ------------------------------------------------------------ bwd_main
constexpr int kBwdThreads = 448;
constexpr uint32_t kTileBytes = 32768;
constexpr uint32_t kSmK = 0, kSmV = 32768, kSmQ = 65536, kSmDO = 131072, kSmDS = 196608;
constexpr uint32_t kBwdSmem = kSmDS + kTileBytes + 1024;

// TMEM columns.  P^T of q-rows [64h, 64h+64) is packed into S^T columns
// [64h, 64h+32) and dS^T into dP^T columns [128+64h, 128+64h+32), so each
// compute half only overwrites S^T / dP^T columns it has already read.
constexpr uint32_t kTmS = 0, kTmDP = 128, kTmDV = 256, kTmDK = 384;
constexpr uint32_t kTmP = 0, kTmDST = 128, kTmDQ = 128;
// A-operand column of k-step kk (q-rows 16kk..16kk+15) for P^T / dS^T.
__device__ __forceinline__ uint32_t ts_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

struct BwdBars {
  uint64_t kv_full, kv_empty, qdo_full[2], qdo_empty[2], sdp_full, pds_full[2], dk_done, dv_done,
      dq_full, dq_free, dkv_free, fin;
};

struct BwdParams {
  msa_plan plan;
  const float* lse;
  const float* delta;
  void* dq_pool;
  float* dk_pool;
  float* dv_pool;
  float c2;     // scale * log2(e)
  float scale;
  int chunk;
  int dq_accum;
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
// Task record i of this CTA's walk, or an empty record past the end.
__device__ __forceinline__ int4 task_rec(const int4* tasks, int64_t i, int64_t n, int chunk) {
  return i < n ? tasks[cta_task(i, chunk)] : make_int4(0, 0, 1 << 8, -1);
}
__device__ __forceinline__ int32_t task_token(const int32_t* col, const TaskView& tv, int qi) {
  return col[tv.col_begin + (qi < tv.nq ? qi : tv.nq - 1)];
}

// MMA issuer of k_bwd_main (one thread).  A function of its own so its few
// live values stay in registers whatever the compute roles need.
//
// Per task t (waits in brackets):
//   [dq_free(t-1)] dP^T(t)  [pds_0] dK, dV k-steps of q-rows 0-63
//   [pds_1] dK, dV k-steps of q-rows 64-127  [dk_done] dQ^T(t)  [dv_done] S^T(t+1)
// so the GEMMs of the first half overlap the softmax of the second.
__device__ __noinline__ void bwd_mma_role(BwdBars& bars, uint32_t tmem, uint32_t sbase,
                                          const int4* tasks, int64_t my_n, int chunk,
                                          volatile int* abort_flag) {
  constexpr uint32_t idKK = idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T
  constexpr uint32_t idTS = idesc_bf16_f32(128, 128, 0, 1);  // dV, dK (A in TMEM)
  constexpr uint32_t idMM = idesc_bf16_f32(128, 128, 1, 1);  // dQ^T
  auto wait = [&](uint64_t& bar, uint32_t ph) {
    const bool ok = mbar_wait(smem_u32(&bar), ph, abort_flag);
    tc_fence_after();
    return ok;
  };
  // Descriptors are built once; a k-step only adds a constant to the
  // start-address field (addresses stay below 256 KB, so the 14-bit field
  // never carries).  Rebuilding a descriptor per MMA costs more issue time
  // than a 128x128x16 MMA takes to run.
  const uint64_t kK = sdesc_sw128(sbase + kSmK, 16u, 1024u);       // K, K-major
  const uint64_t kV = sdesc_sw128(sbase + kSmV, 16u, 1024u);       // V, K-major
  const uint64_t mK = sdesc_sw128(sbase + kSmK, 16384u, 1024u);    // K, MN-major
  const uint64_t mDS = sdesc_sw128(sbase + kSmDS, 16384u, 1024u);  // dS, MN-major
  const uint64_t kQ0 = sdesc_sw128(sbase + kSmQ, 16u, 1024u);
  const uint64_t kDO0 = sdesc_sw128(sbase + kSmDO, 16u, 1024u);
  const uint64_t mQ0 = sdesc_sw128(sbase + kSmQ, 16384u, 1024u);
  const uint64_t mDO0 = sdesc_sw128(sbase + kSmDO, 16384u, 1024u);
  constexpr uint64_t kStage = kTileBytes >> 4;
  // start-address steps (16-byte units): K-major k-step, MN-major k-step
  auto kstep = [](int kk) { return uint64_t((kk >> 2) * 1024 + (kk & 3) * 2); };
  auto mstep = [](int kk) { return uint64_t(kk) * 128u; };
  auto issue_S = [&](int64_t t) {
    const uint64_t b = kQ0 + uint64_t(t & 1) * kStage;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ss(tmem + kTmS, kK + kstep(kk), b + kstep(kk), idKK, kk > 0);
  };
  auto issue_dP = [&](int64_t t) {
    const uint64_t b = kDO0 + uint64_t(t & 1) * kStage;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ss(tmem + kTmDP, kV + kstep(kk), b + kstep(kk), idKK, kk > 0);
    umma_commit(smem_u32(&bars.sdp_full));
  };
  // dK += dS^T Q and dV += P^T dO over the four k-steps of one half of the q-rows
  auto issue_dkdv = [&](int64_t t, int h, uint32_t acc0) {
    const uint64_t bq = mQ0 + uint64_t(t & 1) * kStage;
    const uint64_t bo = mDO0 + uint64_t(t & 1) * kStage;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      umma_ts(tmem + kTmDK, tmem + kTmDST + ts_col(4 * h + j), bq + mstep(4 * h + j), idTS,
              j > 0 ? 1u : acc0);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      umma_ts(tmem + kTmDV, tmem + kTmP + ts_col(4 * h + j), bo + mstep(4 * h + j), idTS,
              j > 0 ? 1u : acc0);
  };
  int64_t kv_loads = 1, seg_done = 0;
  bool first_in_seg = true;
  int cur_kv = task_rec(tasks, 0, my_n, chunk).w;
  int next_kv = task_rec(tasks, 1, my_n, chunk).w;
  bool ok = wait(bars.kv_full, 0) && wait(bars.qdo_full[0], 0);
  if (ok) issue_S(0);
  for (int64_t it = 0; ok && it < my_n; ++it) {
    const uint32_t ph = uint32_t(it & 1);
    const int next2_kv = task_rec(tasks, it + 2, my_n, chunk).w;  // used next iteration
    // dP^T(it) overwrites dQ^T(it-1): the reducers must have read it.
    if (it >= 1 && !wait(bars.dq_free, ph ^ 1u)) break;
    issue_dP(it);
    if (!wait(bars.pds_full[0], ph)) break;
    if (first_in_seg && seg_done > 0 && !wait(bars.dkv_free, uint32_t((seg_done - 1) & 1)))
      break;
    issue_dkdv(it, 0, first_in_seg ? 0u : 1u);
    if (!wait(bars.pds_full[1], ph)) break;
    issue_dkdv(it, 1, 1u);
    umma_commit(smem_u32(&bars.dk_done));
    umma_commit(smem_u32(&bars.dv_done));
    // dQ^T is written over dS^T: dK must have read it.
    if (!wait(bars.dk_done, ph)) break;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ss(tmem + kTmDQ, mK + mstep(kk), mDS + mstep(kk), idMM, kk > 0);
    umma_commit(smem_u32(&bars.dq_full));
    first_in_seg = false;
    if (it + 1 < my_n) {
      if (next_kv != cur_kv) {
        ++seg_done;
        umma_commit(smem_u32(&bars.kv_empty));
        if (!wait(bars.kv_full, uint32_t(kv_loads & 1))) break;
        ++kv_loads;
        cur_kv = next_kv;
        first_in_seg = true;
      }
      // S^T(it+1) overwrites P^T(it): dV(it) must have read it.
      if (!wait(bars.dv_done, ph)) break;
      if (!wait(bars.qdo_full[(it + 1) & 1], uint32_t(((it + 1) >> 1) & 1))) break;
      issue_S(it + 1);
    }
    next_kv = next2_kv;
  }
  umma_commit(smem_u32(&bars.fin));
  mbar_wait_drain(smem_u32(&bars.fin), 0);
}

// Warp roles (448 threads):
//   0      TMA producer: K/V per block run, Q/dO per task (two stages)
//   1      MMA issuer, TMEM owner
//   2-9    compute: P^T, dS^T; warps 2-5 own q-rows [0,64), warps 6-9 [64,128)
//   10-13  reduce: dQ^T -> pool (thread = head dim), dV / dK flush
template <int ACC>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_bwd_main(const __grid_constant__ BwdParams prm, const __grid_constant__ CUtensorMap mapQ,
               const __grid_constant__ CUtensorMap mapDO, const __grid_constant__ CUtensorMap mapK,
               const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapDQ) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, skip_sh;
  __shared__ __align__(16) float s_nlse2[128];  // -LSE * log2(e)
  __shared__ __align__(16) float s_delta[128];
  __shared__ __align__(16) int8_t s_jlim[128];
  __shared__ int s_wfull[4];  // per lane quadrant: every column sees all 128 keys
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
      mbar_init(smem_u32(&bars.qdo_full[i]), 1);
      mbar_init(smem_u32(&bars.qdo_empty[i]), 1);
    }
    mbar_init(smem_u32(&bars.sdp_full), 1);
    mbar_init(smem_u32(&bars.pds_full[0]), 128);
    mbar_init(smem_u32(&bars.pds_full[1]), 128);
    mbar_init(smem_u32(&bars.dk_done), 1);
    mbar_init(smem_u32(&bars.dv_done), 1);
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
  const int chunk = prm.chunk;

  if (warp == 0) {
    // ---------------- TMA producer (task records and tokens prefetched one task ahead)
    if (lane == 0 && my_n > 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapDO);
      tma_prefetch_desc(&mapK);
      tma_prefetch_desc(&mapV);
      int prev_kv = -1;
      int64_t kv_loads = 0, it = 0;
      int4 rec = task_rec(tasks, 0, my_n, chunk), rec1 = task_rec(tasks, 1, my_n, chunk);
      int32_t tok[kTaskQueries];
      {
        const TaskView tv = decode_task(rec);
#pragma unroll
        for (int qi = 0; qi < kTaskQueries; ++qi) tok[qi] = task_token(p.col, tv, qi);
      }
      for (; it < my_n; ++it) {
        const TaskView tv = decode_task(rec);
        const int4 rec2 = task_rec(tasks, it + 2, my_n, chunk);
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
            !mbar_wait(smem_u32(&bars.qdo_empty[st]), uint32_t(((it >> 1) - 1) & 1), abort_flag))
          break;
        const uint32_t b = smem_u32(&bars.qdo_full[st]);
        mbar_arrive_expect_tx(b, 2 * kTileBytes);
        const uint32_t dq = sbase + kSmQ + st * kTileBytes, dd = sbase + kSmDO + st * kTileBytes;
#pragma unroll
        for (int qi = 0; qi < kTaskQueries; ++qi) {
          const int y = tok[qi] * kQHeads + tv.g * kHeadsPerGroup;
          tma_load_2d(dq + qi * 2048, &mapQ, b, 0, y);
          tma_load_2d(dq + 16384 + qi * 2048, &mapQ, b, 64, y);
          tma_load_2d(dd + qi * 2048, &mapDO, b, 0, y);
          tma_load_2d(dd + 16384 + qi * 2048, &mapDO, b, 64, y);
        }
        rec = rec1;
        rec1 = rec2;
#pragma unroll
        for (int qi = 0; qi < kTaskQueries; ++qi) tok[qi] = tok1[qi];
      }
      if (*abort_flag) {  // let armed copies land before the CTA exits
        if (kv_loads > 0) mbar_wait_drain(smem_u32(&bars.kv_full), uint32_t((kv_loads - 1) & 1));
        for (int64_t j = (it >= 2 ? it - 2 : 0); j < it; ++j)
          mbar_wait_drain(smem_u32(&bars.qdo_full[j & 1]), uint32_t((j >> 1) & 1));
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0 && my_n > 0) bwd_mma_role(bars, tmem, sbase, tasks, my_n, chunk, abort_flag);
  } else if (warp < 10) {
    // ---------------- compute: P^T, dS^T (thread = key; half = block of 64 q-rows)
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;  // key within the block = TMEM lane
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    // One 16-column sub-chunk (q-rows cb .. cb+15, cb = 64 half + 16 sc), in
    // fp32 pairs:  P = 2^(S^T c2 - LSE log2 e),  dS = P (dP^T - delta).
    auto sub_chunk = [&](int sc, const uint32_t (&sv)[16], const uint32_t (&dv)[16], bool full) {
      const int cb = half * 64 + sc * 16;
      const uint4* l4 = reinterpret_cast<const uint4*>(s_nlse2 + cb);
      const uint4* d4 = reinterpret_cast<const uint4*>(s_delta + cb);
      const uint4 jw = *reinterpret_cast<const uint4*>(s_jlim + cb);
      const uint32_t jwa[4] = {jw.x, jw.y, jw.z, jw.w};
      uint64_t nl[8], dl[8];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint4 x = l4[q4], y = d4[q4];
        nl[2 * q4] = f2_pack(x.x, x.y);
        nl[2 * q4 + 1] = f2_pack(x.z, x.w);
        dl[2 * q4] = f2_pack(y.x, y.y);
        dl[2 * q4 + 1] = f2_pack(y.z, y.w);
      }
      const uint64_t cc = f2_pack(__float_as_uint(prm.c2), __float_as_uint(prm.c2));
      uint32_t pp[8], pd[8];
#pragma unroll
      for (int jp = 0; jp < 8; ++jp) {
        const uint64_t x2 = f2_fma(f2_pack(sv[2 * jp], sv[2 * jp + 1]), cc, nl[jp]);
        float p0 = fast_exp2(f2_lo(x2)), p1 = fast_exp2(f2_hi(x2));
        if (!full) {  // keys after the column's query (diagonal block) get P = 0
          const int j = 2 * jp;
          const int jl0 = int(int8_t((jwa[j >> 2] >> (8 * (j & 3))) & 0xFF));
          const int jl1 = int(int8_t((jwa[j >> 2] >> (8 * ((j + 1) & 3))) & 0xFF));
          p0 = r <= jl0 ? p0 : 0.f;
          p1 = r <= jl1 ? p1 : 0.f;
        }
        const uint64_t p2 = f2_pack(__float_as_uint(p0), __float_as_uint(p1));
        const uint64_t ds = f2_mul(p2, f2_sub(f2_pack(dv[2 * jp], dv[2 * jp + 1]), dl[jp]));
        pp[jp] = pack_bf16x2(p0, p1);
        pd[jp] = pack_bf16x2(f2_lo(ds), f2_hi(ds));
      }
      tmem_st8_nc(tmem + lane_base + kTmP + half * 64 + sc * 8, pp);
      tmem_st8_nc(tmem + lane_base + kTmDST + half * 64 + sc * 8, pd);
      // dS (B operand of dQ^T, MN-major): tile row = key r, cols = q-rows
      const uint32_t rowb = sbase + kSmDS + half * 16384 + r * 128;
      const uint32_t c0 = uint32_t((2 * sc) ^ (r & 7)) * 16;
      const uint32_t c1 = uint32_t((2 * sc + 1) ^ (r & 7)) * 16;
      st_shared_v4_nc(rowb + c0, pd[0], pd[1], pd[2], pd[3]);
      st_shared_v4_nc(rowb + c1, pd[4], pd[5], pd[6], pd[7]);
    };
    // Column scalars of task it+1 are loaded while task it is computed, in
    // two steps so no load result is consumed right after it is issued: the
    // column's token at the top of task it, its LSE / delta mid-way.
    const int qi = r >> 4, hh = r & 15;
    int4 rec1 = task_rec(tasks, 1, my_n, chunk);
    // (raw LSE: scaling it where it is loaded would wait for the load)
    float clse = 0.f, cdl = 0.f;  // current task's column values
    int cjl = -1;
    if (half == 0 && my_n > 0) {
      const TaskView tv = decode_task(task_rec(tasks, 0, my_n, chunk));
      const int32_t tok = task_token(p.col, tv, qi);
      const int64_t grow = int64_t(tok) * kQHeads + tv.g * kHeadsPerGroup + hh;
      cjl = qi < tv.nq ? min(tok - tv.key_start, tv.key_len - 1) : -1;
      clse = prm.lse[grow];
      cdl = prm.delta[grow];
    }
    for (int64_t it = 0; it < my_n; ++it) {
      const int4 rec2 = task_rec(tasks, it + 2, my_n, chunk);
      int32_t ntok = 0;
      if (half == 0 && it + 1 < my_n) ntok = task_token(p.col, decode_task(rec1), qi);
      named_bar_sync(1, 256);  // previous task's columns fully consumed
      if (half == 0) {
        s_nlse2[r] = -clse * kLog2e;
        s_delta[r] = cdl;
        s_jlim[r] = int8_t(cjl);
        const bool wf = __all_sync(0xffffffffu, cjl == kBlock - 1);
        if (lane == 0) s_wfull[quad] = wf ? 1 : 0;
      }
      named_bar_sync(1, 256);
      if (!mbar_wait_warp(smem_u32(&bars.sdp_full), uint32_t(it & 1), abort_flag)) break;
      tc_fence_after();
      const bool full = s_wfull[0] & s_wfull[1] & s_wfull[2] & s_wfull[3];
      const uint32_t cS = tmem + lane_base + kTmS + half * 64;
      const uint32_t cD = tmem + lane_base + kTmDP + half * 64;
      uint32_t sA[16], dA[16], sB[16], dB[16];
      tmem_ld16(cS, sA);
      tmem_ld16(cD, dA);
      tmem_ld_wait();
#pragma unroll 1
      for (int sp = 0; sp < 2; ++sp) {
        const int sc0 = 2 * sp, sc1 = 2 * sp + 1;
        tmem_ld16(cS + sc1 * 16, sB);
        tmem_ld16(cD + sc1 * 16, dB);
        sub_chunk(sc0, sA, dA, full);
        tmem_ld_wait();
        if (sp < 1) {
          tmem_ld16(cS + (sc1 + 1) * 16, sA);
          tmem_ld16(cD + (sc1 + 1) * 16, dA);
          if (half == 0 && it + 1 < my_n) {  // next task's column values
            const TaskView tn = decode_task(rec1);
            const int64_t grow = int64_t(ntok) * kQHeads + tn.g * kHeadsPerGroup + hh;
            cjl = qi < tn.nq ? min(ntok - tn.key_start, tn.key_len - 1) : -1;
            clse = prm.lse[grow];
            cdl = prm.delta[grow];
          }
        }
        sub_chunk(sc1, sB, dB, full);
        tmem_ld_wait();
      }
      tmem_st_wait();
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(smem_u32(&bars.pds_full[half]));
      rec1 = rec2;
    }
  } else {
    // ---------------- reduce: dQ^T -> pool (thread = head dim), dV / dK flush
    const int quad = warp & 3;
    const int d = quad * 32 + lane;  // head dim = TMEM lane (dQ^T); key for dV / dK
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    const bool odd = lane & 1;
    const bool issuer = (warp == 10 && lane == 0);
    int4 rec = task_rec(tasks, 0, my_n, chunk), rec1 = task_rec(tasks, 1, my_n, chunk);
    for (int64_t it = 0; it < my_n; ++it) {
      const TaskView tv = decode_task(rec);
      const int4 rec2 = task_rec(tasks, it + 2, my_n, chunk);
      int32_t tok[kTaskQueries];
#pragma unroll
      for (int qi = 0; qi < kTaskQueries; ++qi) tok[qi] = task_token(p.col, tv, qi);
      if (!mbar_wait_warp(smem_u32(&bars.dq_full), uint32_t(it & 1), abort_flag)) break;
      tc_fence_after();
      const int64_t gb = int64_t(tv.g) * kHeadsPerGroup;
      const int st = int(it & 1);
      // dq_full(it) means every MMA of the task is complete, so the task's
      // Q tile is free: stage the 16-bit dQ tile row-major in it, then one
      // thread adds it to the pool with one bulk tensor reduction per query
      // (16 heads x 128 dims = 4 KB) and hands the Q/dO stage back to the
      // producer.  Even lanes write (row j, dims d, d+1), odd lanes (row j+1,
      // dims d-1, d).
      const uint32_t stage_base = sbase + kSmQ + st * kTileBytes;
      const uint32_t stage = stage_base + uint32_t(odd ? 256 + 2 * (d - 1) : 2 * d);
      auto consume = [&](const uint32_t (&v)[64], int j0) {
        if (ACC == MSA_DQ_ACCUM_F32) {
          float* pool = static_cast<float*>(prm.dq_pool) + d;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            const int jj = j0 + j;
            if ((jj >> 4) < tv.nq)
              red_add_f32(pool + ((int64_t(tok[jj >> 4]) * kQHeads + gb + (jj & 15)) * kHeadDim),
                          __uint_as_float(v[j]) * prm.scale);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 64; j += 2) {
            const float a = __uint_as_float(v[j]) * prm.scale;
            const float b = __uint_as_float(v[j + 1]) * prm.scale;
            const float x = __shfl_xor_sync(0xffffffffu, odd ? a : b, 1);
            const float lo = odd ? x : a, hi = odd ? b : x;
            const uint32_t w2 =
                ACC == MSA_DQ_ACCUM_F16 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi);
            const int jj = j0 + j;
            st_shared_b32(stage + (jj >> 4) * 4096 + (jj & 15) * 256, w2);
          }
        }
      };
      uint32_t v[64];
      tmem_ld32(tmem + lane_base + kTmDQ + 0, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(tmem + lane_base + kTmDQ + 32, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait();
      consume(v, 0);
      tmem_ld32(tmem + lane_base + kTmDQ + 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(tmem + lane_base + kTmDQ + 96, *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.dq_free));
      consume(v, 64);
      if (ACC != MSA_DQ_ACCUM_F32) {
        fence_proxy_async_smem();
        named_bar_sync(2, 128);
        if (issuer) {
          for (int qi = 0; qi < tv.nq; ++qi)
            for (unsigned h0 = 0; h0 < unsigned(kHeadsPerGroup); h0 += kDqReduceRows)
              tma_reduce_add_2d(&mapDQ, stage_base + qi * 4096 + h0 * 256, 0,
                                tok[qi] * kQHeads + tv.g * kHeadsPerGroup + int(h0));
          bulk_commit();
          bulk_wait_read0();
          mbar_arrive(smem_u32(&bars.qdo_empty[st]));
        }
      } else if (issuer) {
        mbar_arrive(smem_u32(&bars.qdo_empty[st]));
      }
      const bool seg_end = (it + 1 == my_n) || rec1.w != tv.sub;
      if (seg_end) {
        // dq_full(it) follows dv_done / dk_done(it): dV / dK of the run are final.
        const int key = d;
        const bool key_valid = key < tv.key_len;
        const int64_t krow = (int64_t(tv.key_start) + key) * kKVHeads + tv.g;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t a[32], b[32];
          tmem_ld32(tmem + lane_base + kTmDV + c * 32, a);
          tmem_ld32(tmem + lane_base + kTmDK + c * 32, b);
          tmem_ld_wait();
          if (key_valid) {
            float* dvr = prm.dv_pool + krow * kHeadDim + c * 32;
            float* dkr = prm.dk_pool + krow * kHeadDim + c * 32;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
              red_add_v4_f32(dvr + e, __uint_as_float(a[e]), __uint_as_float(a[e + 1]),
                             __uint_as_float(a[e + 2]), __uint_as_float(a[e + 3]));
              red_add_v4_f32(dkr + e, __uint_as_float(b[e]) * prm.scale,
                             __uint_as_float(b[e + 1]) * prm.scale,
                             __uint_as_float(b[e + 2]) * prm.scale,
                             __uint_as_float(b[e + 3]) * prm.scale);
            }
          }
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.dkv_free));
      }
      rec = rec1;
      rec1 = rec2;
    }
    if (issuer) bulk_wait0();  // bulk reductions complete before the CTA exits
  }

  if (threadIdx.x == 0 && abort_sh) raise_status(p.header, MSA_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ bwd_finalize
// Pools -> bf16 outputs, 8 elements per thread.
__global__ void __launch_bounds__(256) k_bwd_finalize(msa_plan p, const void* dq_pool,
                                                      const float* dk_pool, const float* dv_pool,
                                                      __nv_bfloat16* dq, __nv_bfloat16* dk,
                                                      __nv_bfloat16* dv) {
  if (plan_failed(p.header)) return;
  const int64_t nq8 = p.T * kQHeads * kHeadDim / 8, nk8 = p.T * kKVHeads * kHeadDim / 8;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < nq8 + 2 * nk8;
       i += stride) {
    float f[8];
    uint4* dst;
    if (i < nq8) {
      if (p.dq_accum == MSA_DQ_ACCUM_F32) {
        const float4 a = reinterpret_cast<const float4*>(dq_pool)[2 * i];
        const float4 b = reinterpret_cast<const float4*>(dq_pool)[2 * i + 1];
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
      } else {
        const uint4 a = reinterpret_cast<const uint4*>(dq_pool)[i];
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (p.dq_accum == MSA_DQ_ACCUM_F16) {
            f[2 * e] = f16_lo(w[e]);
            f[2 * e + 1] = f16_hi(w[e]);
          } else {
            f[2 * e] = bf16_lo(w[e]);
            f[2 * e + 1] = bf16_hi(w[e]);
          }
        }
      }
      dst = reinterpret_cast<uint4*>(dq) + i;
    } else {
      const int64_t j = i < nq8 + nk8 ? i - nq8 : i - nq8 - nk8;
      const float* src = i < nq8 + nk8 ? dk_pool : dv_pool;
      const float4 a = reinterpret_cast<const float4*>(src)[2 * j];
      const float4 b = reinterpret_cast<const float4*>(src)[2 * j + 1];
      f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
      f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
      dst = reinterpret_cast<uint4*>(i < nq8 + nk8 ? dk : dv) + j;
    }
    *dst = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
  }
}

}  // namespace

CUresult make_map_rows(CUtensorMap* m, const void* base, int64_t rows);
CUresult make_map_kv(CUtensorMap* m, const void* base, int64_t T);
CUresult make_map_pool16(CUtensorMap* m, const void* base, int64_t rows, bool bf16);
int device_sm_count();

size_t backward_workspace_bytes(const msa_plan& p) { return bwd_layout(p).total; }

cudaError_t launch_backward(const msa_plan& p, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout, float scale,
                            void* dq, void* dk, void* dv, void* ws, cudaStream_t s) {
  const BwdLayout L = bwd_layout(p);
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* delta = reinterpret_cast<float*>(w + L.off_delta);
  void* dq_pool = w + L.off_dq;
  float* dk_pool = reinterpret_cast<float*>(w + L.off_dk);
  float* dv_pool = reinterpret_cast<float*>(w + L.off_dv);

  CUtensorMap mQ, mDO, mK, mV, mDQ;
  memset(&mDQ, 0, sizeof mDQ);
  if (make_map_rows(&mQ, q, p.T * kQHeads) != CUDA_SUCCESS ||
      make_map_rows(&mDO, dout, p.T * kQHeads) != CUDA_SUCCESS ||
      make_map_kv(&mK, k, p.T) != CUDA_SUCCESS || make_map_kv(&mV, v, p.T) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if (p.dq_accum != MSA_DQ_ACCUM_F32 &&
      make_map_pool16(&mDQ, dq_pool, p.T * kQHeads, p.dq_accum == MSA_DQ_ACCUM_BF16) !=
          CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  const int64_t rows = p.T * kQHeads;
  const int64_t dq_vec = int64_t(dq_elem_bytes(p)) * rows * kHeadDim / 16;
  // dk and dv pools are contiguous in the workspace (dv follows dk)
  const int64_t dkv_vec = int64_t(L.off_dv - L.off_dk) / 16 + p.T * kKVHeads * kHeadDim / 4;
  const int64_t warps = (rows + kDeltaRowsPerWarp - 1) / kDeltaRowsPerWarp;
  launch_begin("bwd_delta", s);
  k_bwd_delta<<<unsigned((warps + 7) / 8), 256, 0, s>>>(
      p, static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), delta,
      static_cast<uint4*>(dq_pool), dq_vec, reinterpret_cast<float4*>(dk_pool), dkv_vec);
  launch_end("bwd_delta", s);

  static bool attr_set = false;
  if (!attr_set) {
    for (auto fn : {k_bwd_main<MSA_DQ_ACCUM_F16>, k_bwd_main<MSA_DQ_ACCUM_BF16>,
                    k_bwd_main<MSA_DQ_ACCUM_F32>}) {
      cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
      if (e != cudaSuccess) return e;
    }
    attr_set = true;
  }
  BwdParams prm{p, lse, delta, dq_pool, dk_pool, dv_pool, scale * kLog2e, scale, 64,
                p.dq_accum};
  launch_begin("bwd_main", s);
  const unsigned grid = unsigned(device_sm_count());
  if (p.dq_accum == MSA_DQ_ACCUM_F32)
    k_bwd_main<MSA_DQ_ACCUM_F32><<<grid, kBwdThreads, kBwdSmem, s>>>(prm, mQ, mDO, mK, mV, mDQ);
  else if (p.dq_accum == MSA_DQ_ACCUM_BF16)
    k_bwd_main<MSA_DQ_ACCUM_BF16><<<grid, kBwdThreads, kBwdSmem, s>>>(prm, mQ, mDO, mK, mV, mDQ);
  else
    k_bwd_main<MSA_DQ_ACCUM_F16><<<grid, kBwdThreads, kBwdSmem, s>>>(prm, mQ, mDO, mK, mV, mDQ);
  launch_end("bwd_main", s);
  launch_begin("bwd_finalize", s);
  k_bwd_finalize<<<unsigned(device_sm_count() * 8), 256, 0, s>>>(
      p, dq_pool, dk_pool, dv_pool, static_cast<__nv_bfloat16*>(dq),
      static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv));
  launch_end("bwd_finalize", s);
  return cudaGetLastError();
}

}  // namespace msa
