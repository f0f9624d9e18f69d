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
// per key; lane = head dimension for dQ^T, so a thread holds one head
// dimension of all the task's query heads.  dV / dK accumulate over a run of
// tasks that share the K/V block and are flushed with fp32 L2 reductions.
// dQ goes straight from registers into a pool interleaved by head octets
// (the eight heads 8o..8o+7 of a token side by side per head dimension) with
// 16-byte packed atomics (fp16 by default, bf16 or fp32 on request): a
// warp-wide atomic covers 512 contiguous bytes, and no shared memory is
// involved.  A warp issues such atomics only one every ~200 cycles, so the
// twelve warps that can reach a TMEM lane quadrant share them: the eight
// compute warps take the first 32 q-rows of their half, the four flush warps
// the other 32 of each half.
//
// bwd_main runs 14 warps: a TMA producer, an MMA issuer, eight compute warps
// (P^T, dS^T, dQ^T readout; two per TMEM lane quadrant, each owning 64
// q-rows) and four warps that flush dV / dK at the end of each run.
//
// Kernels, in launch order:
//   bwd_delta     delta = rowsum(dO * O); zero the dQ / dK / dV pools
//   bwd_main      the tensor-core tile loop
//   bwd_finalize  pools -> bf16 dQ (de-interleaved), dK, dV
#include "common.cuh"
#include "sm100.cuh"

#include <cstring>
#include <type_traits>

namespace msa {

#ifdef MSA_TEST_STARVE
// Test-only build: when set (3), CTA 0 of bwd_main leaves out its first
// Q / dO tiles, so that a bounded wait runs out and the call reports
// MSA_ERR_TIMEOUT.  Set by msa_test_starve.
__device__ int g_starve_bwd;
cudaError_t test_set_starve_bwd(int which) {
  return cudaMemcpyToSymbol(g_starve_bwd, &which, sizeof which);
}
#endif

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
  grid_dep_wait();
  grid_dep_release();
  // the range warning describes one backward: start this one without it
  if (blockIdx.x == 0 && threadIdx.x == 0) clear_warnings(p.header);
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

// TMEM columns.  S^T goes to [0,128).  For the q-rows [64h, 64h+64) of
// compute half h, P^T is packed (bf16 pairs) into S^T columns [64h, 64h+32)
// and dS^T into [64h+32, 64h+64): each half only overwrites S^T columns it
// has already read.  dP^T goes to [128,256) and, once the compute warps have
// read it, dQ^T of the same task.  dV and dK accumulate in [256,384) and
// [384,512) over a run of tasks on one key block.
constexpr uint32_t kTmS = 0, kTmDP = 128, kTmDV = 256, kTmDK = 384;
constexpr uint32_t kTmP = 0, kTmDS = 32, kTmDQ = 128;
// A-operand column of k-step kk (q-rows 16kk..16kk+15) for P^T (add kTmDS
// for dS^T).
__device__ __forceinline__ uint32_t ts_col(int kk) { return (kk >> 2) * 64 + (kk & 3) * 8; }

struct BwdBars {
  uint64_t kv_full, kv_empty, qdo_full[2], qdo_empty[2], s_full, dp_full, p_ready[2],
      ds_ready[2], pt_free, dq_full, dq_free, seg_done, dkv_free, cols, fin;
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
  int dq_accum;
};

// Tasks per chunk of the CTA walk (TaskWalk: full rounds of chunks go
// round-robin over the CTAs, the rest is split evenly).
constexpr int kBwdChunk = 64;
// Task record i of this CTA's walk; past the end, the last one (every
// caller guards its uses by the index).  Only the address depends on the
// index test, never the loaded value, so nothing waits for the load until
// the record is used.  With no tasks, entry 0 of the (allocated) table.
__device__ __forceinline__ int4 task_rec(const int4* tasks, int64_t i, const TaskWalk& w) {
  return tasks[w.n > 0 ? walk_task<kBwdChunk>(w, i < w.n ? i : w.n - 1) : 0];
}
__device__ __forceinline__ int32_t task_token(const int32_t* col, const TaskView& tv, int qi) {
  return col[tv.col_begin + (qi < tv.nq ? qi : tv.nq - 1)];
}

// MMA issuer of k_bwd_main (one thread).  A function of its own so its few
// live values stay in registers whatever the compute roles need.
//
// Issue order for task t (waits in brackets):
//   S^T(t), dP^T(t)                          (issued at the end of task t-1)
//   [p_ready 0] dV k-steps of q-rows 0-63   [p_ready 1] q-rows 64-127
//   [ds_ready 0] dK k-steps of q-rows 0-63  [ds_ready 1] q-rows 64-127
//   dQ^T(t) into the dP^T columns (the compute warps have read dP^T(t))
//   [pt_free] S^T(t+1)  [dq_free] dP^T(t+1)
// The compute warps exponentiate S^T(t) while dP^T(t) runs, dV(t) starts as
// soon as P^T(t) is in TMEM, and the compute warps read dQ^T(t) out while
// S^T(t+1) runs.
__device__ __noinline__ void bwd_mma_role(BwdBars& bars, uint32_t tmem, uint32_t sbase,
                                          const int4* tasks, const TaskWalk walk,
                                          volatile int* abort_flag) {
  const int64_t my_n = walk.n;
  constexpr uint32_t idKK = idesc_bf16_f32(128, 128, 0, 0);  // S^T, dP^T
  constexpr uint32_t idKM = idesc_bf16_f32(128, 128, 0, 1);  // dV, dK (A in TMEM)
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
    umma_commit(smem_u32(&bars.s_full));
  };
  auto issue_dP = [&](int64_t t) {
    const uint64_t b = kDO0 + uint64_t(t & 1) * kStage;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ss(tmem + kTmDP, kV + kstep(kk), b + kstep(kk), idKK, kk > 0);
    umma_commit(smem_u32(&bars.dp_full));
  };
  // dV += P^T dO over the four k-steps of one half of the q-rows
  auto issue_dv = [&](int64_t t, int h, uint32_t acc0) {
    const uint64_t bo = mDO0 + uint64_t(t & 1) * kStage;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      umma_ts(tmem + kTmDV, tmem + kTmP + ts_col(4 * h + j), bo + mstep(4 * h + j), idKM,
              j > 0 ? 1u : acc0);
  };
  // dK += dS^T Q over the four k-steps of one half of the q-rows
  auto issue_dk = [&](int64_t t, int h, uint32_t acc0) {
    const uint64_t bq = mQ0 + uint64_t(t & 1) * kStage;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      umma_ts(tmem + kTmDK, tmem + kTmP + kTmDS + ts_col(4 * h + j), bq + mstep(4 * h + j), idKM,
              j > 0 ? 1u : acc0);
  };
  int64_t kv_loads = 1, seg_done = 0;
  bool first_in_seg = true;
  int cur_kv = task_rec(tasks, 0, walk).w;
  int next_kv = task_rec(tasks, 1, walk).w;
  bool ok = wait(bars.kv_full, 0) && wait(bars.qdo_full[0], 0);
  if (ok) {
    issue_S(0);
    issue_dP(0);
  }
  for (int64_t it = 0; ok && it < my_n; ++it) {
    const uint32_t ph = uint32_t(it & 1);
    const int next2_kv = task_rec(tasks, it + 2, walk).w;  // used next iteration
    const uint32_t acc0 = first_in_seg ? 0u : 1u;
    // the first dV / dK of a run overwrite the accumulators: the reducers
    // must have flushed the previous run
    if (first_in_seg && seg_done > 0 && !wait(bars.dkv_free, uint32_t((seg_done - 1) & 1)))
      break;
    if (!wait(bars.p_ready[0], ph)) break;
    issue_dv(it, 0, acc0);
    if (!wait(bars.p_ready[1], ph)) break;
    issue_dv(it, 1, 1u);
    if (!wait(bars.ds_ready[0], ph)) break;
    issue_dk(it, 0, acc0);
    if (!wait(bars.ds_ready[1], ph)) break;
    issue_dk(it, 1, 1u);
    umma_commit(smem_u32(&bars.pt_free));
    // dQ^T into the dP^T columns, which the compute warps have read
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      umma_ss(tmem + kTmDQ, mK + mstep(kk), mDS + mstep(kk), idMM, kk > 0);
    umma_commit(smem_u32(&bars.dq_full));
    first_in_seg = false;
    const bool seg_end = it + 1 == my_n || next_kv != cur_kv;
    if (seg_end) umma_commit(smem_u32(&bars.seg_done));  // dV / dK of the run are final
    if (it + 1 < my_n) {
      if (seg_end) {
        ++seg_done;
        umma_commit(smem_u32(&bars.kv_empty));
        if (!wait(bars.kv_full, uint32_t(kv_loads & 1))) break;
        ++kv_loads;
        cur_kv = next_kv;
        first_in_seg = true;
      }
      // S^T(it+1) overwrites P^T(it) and dS^T(it): dV(it) and dK(it) must
      // have read them.
      if (!wait(bars.pt_free, ph)) break;
      if (!wait(bars.qdo_full[(it + 1) & 1], uint32_t(((it + 1) >> 1) & 1))) break;
      issue_S(it + 1);
      // dP^T(it+1) overwrites dQ^T(it): the reducers must have read it.
      if (!wait(bars.dq_free, ph)) break;
      issue_dP(it + 1);
    }
    next_kv = next2_kv;
  }
  umma_commit(smem_u32(&bars.fin));
  mbar_wait_drain(smem_u32(&bars.fin), 0);
}

// Adds dQ^T of two queries (q0, q0+1 of the task; 32 q-rows = 4 head octets,
// values v of head dimension d) to the octet-interleaved pool: one 16-byte
// packed atomic per octet (two for fp32).
template <int ACC>
__device__ __forceinline__ void dq_atomics(const BwdParams& prm, const uint32_t (&v)[32],
                                           const int32_t (&tok)[2], const TaskView& tv, int q0,
                                           int d) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (q0 + k >= tv.nq) continue;
    const int64_t oct0 = int64_t(tok[k]) * (kQHeads / 8) + tv.g * (kHeadsPerGroup / 8);
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = __uint_as_float(v[16 * k + 8 * o + e]) * prm.scale;
      const int64_t el = ((oct0 + o) * kHeadDim + d) * 8;
      if (ACC == MSA_DQ_ACCUM_F32) {
        float* dst = static_cast<float*>(prm.dq_pool) + el;
        red_add_v4_f32(dst, x[0], x[1], x[2], x[3]);
        red_add_v4_f32(dst + 4, x[4], x[5], x[6], x[7]);
      } else if (ACC == MSA_DQ_ACCUM_BF16) {
        red_add_v4_bf16x2(static_cast<uint16_t*>(prm.dq_pool) + el, pack_bf16x2(x[0], x[1]),
                          pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]),
                          pack_bf16x2(x[6], x[7]));
      } else {
        red_add_v4_f16x2(static_cast<uint16_t*>(prm.dq_pool) + el, pack_f16x2(x[0], x[1]),
                         pack_f16x2(x[2], x[3]), pack_f16x2(x[4], x[5]),
                         pack_f16x2(x[6], x[7]));
      }
    }
  }
}

// Warp roles (448 threads):
//   0      TMA producer: K/V per block run, Q/dO per task (two stages)
//   1      MMA issuer, TMEM owner
//   2-9    compute: P^T, dS^T (TMEM) and dS (shared memory), then dQ^T of
//          q-rows [64h, 64h+32) read out of TMEM and added to the pool with
//          packed atomics; warps 2-5 own q-rows [0,64) (h = 0), warps 6-9
//          [64,128) (h = 1)
//   10-13  dQ^T of q-rows [32,64) and [96,128) (thread = head dim); dV / dK
//          flush at the end of a run (thread = key)
template <int ACC>
__global__ void __launch_bounds__(kBwdThreads, 1)
    k_bwd_main(const __grid_constant__ BwdParams prm, const __grid_constant__ CUtensorMap mapQ,
               const __grid_constant__ CUtensorMap mapDO, const __grid_constant__ CUtensorMap mapK,
               const __grid_constant__ CUtensorMap mapV) {
  grid_dep_wait();
  grid_dep_release();
  extern __shared__ uint8_t smem_raw[];
  __shared__ BwdBars bars;
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_sh, skip_sh;
  // Column (q-row) scalars of the current task.
  __shared__ __align__(16) float s_nlse2[128];  // -LSE * log2(e)
  __shared__ __align__(16) float s_delta[128];
  __shared__ __align__(16) int8_t s_jlim[128];  // last visible key, -1 for padding
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
    mbar_init(smem_u32(&bars.s_full), 1);
    mbar_init(smem_u32(&bars.dp_full), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars.p_ready[i]), 128);
      mbar_init(smem_u32(&bars.ds_ready[i]), 128);
    }
    mbar_init(smem_u32(&bars.pt_free), 1);
    mbar_init(smem_u32(&bars.dq_full), 1);
    mbar_init(smem_u32(&bars.dq_free), 384);
    mbar_init(smem_u32(&bars.seg_done), 1);
    mbar_init(smem_u32(&bars.dkv_free), 128);
    mbar_init(smem_u32(&bars.cols), 256);
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
  const TaskWalk walk = task_walk<kBwdChunk>(ntasks);
  const int64_t my_n = walk.n;
  const int4* tasks = reinterpret_cast<const int4*>(p.tasks);

  if (warp == 0) {
    // ---------------- TMA producer (task records and tokens prefetched one task ahead)
    if (lane == 0 && my_n > 0) {
      tma_prefetch_desc(&mapQ);
      tma_prefetch_desc(&mapDO);
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
#ifdef MSA_TEST_STARVE
        if (!(g_starve_bwd == 3 && blockIdx.x == 0 && it == 0)) {
#endif
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
#ifdef MSA_TEST_STARVE
        }
#endif
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
    if (lane == 0 && my_n > 0) bwd_mma_role(bars, tmem, sbase, tasks, walk, abort_flag);
  } else if (warp < 10) {
    // ---------------- compute (thread = TMEM lane; half = block of 64 q-rows)
    // Phase 1 (after S^T; thread = key): P = 2^(S^T c2 - LSE log2 e), masked
    // after the column's query on diagonal blocks, as bf16 pairs into TMEM
    // (A operand of dV) and kept in registers.  Phase 2 (after dP^T):
    // dS = P (dP^T - delta) as bf16 into TMEM (A operand of dK) and into the
    // shared-memory dS tile (row = key, 128-byte swizzle; B operand of dQ^T).
    // Phase 3 (after dQ^T; thread = head dim): dQ^T of q-rows [64h, 64h+32)
    // (queries 4h, 4h+1) read out, scaled and added to the pool with packed
    // atomics.
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;  // key (phases 1, 2) / head dim (phase 3) = TMEM lane
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    const uint32_t cS = tmem + lane_base + kTmS + half * 64;
    const uint32_t cD = tmem + lane_base + kTmDP + half * 64;
    const uint32_t cQ = tmem + lane_base + kTmDQ + half * 64;
    const uint32_t rowb = sbase + kSmDS + half * 16384 + r * 128;
    const uint64_t cc = f2_pack(__float_as_uint(prm.c2), __float_as_uint(prm.c2));
    // Half 0 also loads the column scalars of the next task: thread r owns
    // column r (query r / 16 of the task, head r % 16).
    const int qi = r >> 4, hh = r & 15;
    auto col_row = [&](const TaskView& tv, int32_t tok) {
      return int64_t(tok) * kQHeads + tv.g * kHeadsPerGroup + hh;
    };
    auto col_jlim = [&](const TaskView& tv, int32_t tok) {
      return qi < tv.nq ? min(tok - tv.key_start, tv.key_len - 1) : -1;
    };
    auto put_cols = [&](float lse, float dl, int jl) {
      s_nlse2[r] = -lse * kLog2e;
      s_delta[r] = dl;
      s_jlim[r] = int8_t(jl);
      const bool wf = __all_sync(0xffffffffu, jl == kBlock - 1);
      if (lane == 0) s_wfull[quad] = wf ? 1 : 0;
    };
    int4 rec0 = task_rec(tasks, 0, walk), rec1 = task_rec(tasks, 1, walk);
    int32_t tok1 = 0;
    if (my_n > 0) {
      tok1 = task_token(p.col, decode_task(rec1), qi);
      if (half == 0) {
        const TaskView tv = decode_task(rec0);
        const int32_t tok = task_token(p.col, tv, qi);
        const int64_t grow = col_row(tv, tok);
        put_cols(prm.lse[grow], prm.delta[grow], col_jlim(tv, tok));
      }
    }
    // Column scalars of a task are published through the `cols` barrier
    // (phase 0: task 0; phase it + 1: task it + 1).  Half 0 overwrites them
    // once both halves have finished phase 2 of task it (ds_ready).
    mbar_arrive(smem_u32(&bars.cols));
    bool cols_ok = mbar_wait_warp(smem_u32(&bars.cols), 0u, abort_flag);
    uint32_t pk[32];  // P of this thread's key for the half's 64 q-rows, bf16 pairs
    // ---- phase 1 over the half's 64 columns (S^T values in a0, a1)
    auto phase1 = [&](auto full_t, const uint32_t (&a0)[32], const uint32_t (&a1)[32],
                      const float* nl, const int8_t* jl) {
      constexpr bool kFull = decltype(full_t)::value;
#pragma unroll
      for (int q4 = 0; q4 < 16; ++q4) {
        const uint32_t* v = q4 < 8 ? &a0[4 * q4] : &a1[4 * (q4 - 8)];
        const uint4 x = *reinterpret_cast<const uint4*>(nl + 4 * q4);
        const uint64_t e0 = f2_fma(f2_pack(v[0], v[1]), cc, f2_pack(x.x, x.y));
        const uint64_t e1 = f2_fma(f2_pack(v[2], v[3]), cc, f2_pack(x.z, x.w));
        float p0 = fast_exp2(f2_lo(e0)), p1 = fast_exp2(f2_hi(e0));
        float p2 = fast_exp2(f2_lo(e1)), p3 = fast_exp2(f2_hi(e1));
        if constexpr (!kFull) {  // keys after the column's query get P = 0
          const uint32_t w = *reinterpret_cast<const uint32_t*>(jl + 4 * q4);
          p0 = r <= int(int8_t(w & 0xFF)) ? p0 : 0.f;
          p1 = r <= int(int8_t((w >> 8) & 0xFF)) ? p1 : 0.f;
          p2 = r <= int(int8_t((w >> 16) & 0xFF)) ? p2 : 0.f;
          p3 = r <= int(int8_t(w >> 24)) ? p3 : 0.f;
        }
        pk[2 * q4] = pack_bf16x2(p0, p1);
        pk[2 * q4 + 1] = pack_bf16x2(p2, p3);
      }
    };
    for (int64_t it = 0; cols_ok && it < my_n; ++it) {
      const uint32_t ph = uint32_t(it & 1);
      const int st = int(it & 1);
      const int4 rec2 = task_rec(tasks, it + 2, walk);
      // The next task's column scalars: loaded now (unconditionally, so no
      // select waits for them here), stored by half 0 after phase 2.
      const TaskView tv1 = decode_task(rec1);
      const int64_t grow1 = col_row(tv1, tok1);
      const float lse1 = prm.lse[grow1];
      const float dl1 = prm.delta[grow1];
      const int jl1 = col_jlim(tv1, tok1);
      const bool full = (s_wfull[0] & s_wfull[1] & s_wfull[2] & s_wfull[3]) != 0;
      const float* nl = &s_nlse2[half * 64];
      const float* dlt = &s_delta[half * 64];
      const int8_t* jl = &s_jlim[half * 64];
      // ---- phase 1
      if (!mbar_wait_warp(smem_u32(&bars.s_full), ph, abort_flag)) break;
      tc_fence_after();
      {
        uint32_t a0[32], a1[32];
        tmem_ld32(cS, a0);
        tmem_ld32(cS + 32, a1);
        tmem_ld_wait();
        reg_fence32(a0);
        reg_fence32(a1);
        if (full)
          phase1(std::true_type{}, a0, a1, nl, jl);
        else
          phase1(std::false_type{}, a0, a1, nl, jl);
      }
      tmem_st32_nc(cS + kTmP, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.p_ready[half]));
      const int32_t tok2 = task_token(p.col, decode_task(rec2), qi);
      // tokens of the queries 4h, 4h+1, for the dQ atomics of phase 3
      const TaskView tv0 = decode_task(rec0);
      int32_t tq[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) tq[k] = task_token(p.col, tv0, 4 * half + k);
      // ---- phase 2
      if (!mbar_wait_warp(smem_u32(&bars.dp_full), ph, abort_flag)) break;
      tc_fence_after();
      {
        // 16 q-rows at a time; the second 32 columns of dP^T are loaded while
        // the first are processed
        auto chunk = [&](int sc, const uint32_t* v) {
          uint32_t pd[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int q4 = 4 * sc + q;
            const uint4 y = *reinterpret_cast<const uint4*>(dlt + 4 * q4);
            const uint32_t w0 = pk[2 * q4], w1 = pk[2 * q4 + 1];
            const uint64_t da = f2_mul(f2_pack(w0 << 16, w0 & 0xFFFF0000u),
                                       f2_sub(f2_pack(v[4 * q], v[4 * q + 1]), f2_pack(y.x, y.y)));
            const uint64_t db = f2_mul(f2_pack(w1 << 16, w1 & 0xFFFF0000u),
                                       f2_sub(f2_pack(v[4 * q + 2], v[4 * q + 3]), f2_pack(y.z, y.w)));
            pd[2 * q] = pack_bf16x2(f2_lo(da), f2_hi(da));
            pd[2 * q + 1] = pack_bf16x2(f2_lo(db), f2_hi(db));
          }
          tmem_st8_nc(cS + kTmDS + sc * 8, pd);
          // dS tile row = key r, columns = q-rows: 16-byte chunks 2 sc, 2 sc + 1
          // of this half, swizzled by (r & 7)
          st_shared_v4_nc(rowb + uint32_t((2 * sc) ^ (r & 7)) * 16, pd[0], pd[1], pd[2], pd[3]);
          st_shared_v4_nc(rowb + uint32_t((2 * sc + 1) ^ (r & 7)) * 16, pd[4], pd[5], pd[6],
                          pd[7]);
        };
        uint32_t b[32];
        tmem_ld32(cD, b);
        tmem_ld_wait();
        reg_fence32(b);
        chunk(0, &b[0]);
        chunk(1, &b[16]);
        tmem_ld32(cD + 32, b);
        tmem_ld_wait();
        reg_fence32(b);
        chunk(2, &b[0]);
        chunk(3, &b[16]);
      }
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars.ds_ready[half]));
      if (half == 0 && it + 1 < my_n) {
        if (!mbar_wait_warp(smem_u32(&bars.ds_ready[0]), ph, abort_flag) ||
            !mbar_wait_warp(smem_u32(&bars.ds_ready[1]), ph, abort_flag))
          break;
        put_cols(lse1, dl1, jl1);
      }
      // next task's column scalars visible, this task's consumed
      mbar_arrive(smem_u32(&bars.cols));
      if (!mbar_wait_warp(smem_u32(&bars.cols), ph ^ 1u, abort_flag)) break;
      // ---- phase 3: dQ^T (lane = head dim d = r, columns = the half's q-rows)
      if (!mbar_wait_warp(smem_u32(&bars.dq_full), ph, abort_flag)) break;
      tc_fence_after();
      // every MMA of the task is complete: its Q / dO stage is free
      if (warp == 2 && lane == 0) mbar_arrive(smem_u32(&bars.qdo_empty[st]));
      {
        uint32_t v0[32];
        tmem_ld32(cQ, v0);
        tmem_ld_wait();
        reg_fence32(v0);
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.dq_free));  // dP^T(it+1) may overwrite dQ^T(it)
        dq_atomics<ACC>(prm, v0, tq, tv0, 4 * half, r);
      }
      rec0 = rec1;
      rec1 = rec2;
      tok1 = tok2;
    }
  } else {
    // ---------------- dQ^T of q-rows [32,64) and [96,128) (thread = head
    // dim), dV / dK flush at the end of each run (thread = key)
    const int quad = warp & 3;
    const int key = quad * 32 + lane;
    const uint32_t lane_base = uint32_t(quad * 32) << 16;
    int4 rec = task_rec(tasks, 0, walk), rec1 = task_rec(tasks, 1, walk);
    int64_t nseg = 0;
    for (int64_t it = 0; it < my_n; ++it) {
      const TaskView tv = decode_task(rec);
      const int4 rec2 = task_rec(tasks, it + 2, walk);
      int32_t ta[2], tb[2];  // tokens of queries 2, 3 and 6, 7
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        ta[k] = task_token(p.col, tv, 2 + k);
        tb[k] = task_token(p.col, tv, 6 + k);
      }
      if (!mbar_wait_warp(smem_u32(&bars.dq_full), uint32_t(it & 1), abort_flag)) break;
      tc_fence_after();
      {
        uint32_t va[32], vb[32];
        tmem_ld32(tmem + lane_base + kTmDQ + 32, va);
        tmem_ld32(tmem + lane_base + kTmDQ + 96, vb);
        tmem_ld_wait();
        reg_fence32(va);
        reg_fence32(vb);
        tc_fence_before();
        mbar_arrive(smem_u32(&bars.dq_free));
        dq_atomics<ACC>(prm, va, ta, tv, 2, key);
        dq_atomics<ACC>(prm, vb, tb, tv, 6, key);
      }
      const bool seg_end = (it + 1 == my_n) || rec1.w != tv.sub;
      if (seg_end) {
        // seg_done follows the run's last dV / dK MMAs: the accumulators are final
        if (!mbar_wait_warp(smem_u32(&bars.seg_done), uint32_t(nseg & 1), abort_flag)) break;
        ++nseg;
        tc_fence_after();
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
  }

  if (threadIdx.x == 0 && abort_sh) raise_status(p.header, MSA_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ------------------------------------------------------------ bwd_finalize
// Pools -> bf16 outputs.  A 16-bit dQ pool (fp16 default, bf16) is taken a
// head octet of a token at a time: the octet's 2 KB ([128 d][8 heads]) is
// read by one warp, 512 contiguous bytes per instruction, converted and
// transposed through shared memory to [8 heads][128 d], and written back as
// 512 contiguous bytes per instruction.  An fp32 pool: one thread per
// (head octet, 8 head dimensions).  dK / dV: one 128-byte pool line (32
// elements) per thread.  Pool lines of the 16-bit dQ pool and of the dK / dV
// pools are dropped from L2 once read (the pools are zeroed again before
// their next use).  A non-finite value in an fp16 pool (fp16 saturates above
// 65504) sets MSA_ERR_RANGE.
constexpr int kFinThreads = 256;
constexpr int kFinOcts = 2;  // head octets per warp iteration (loads in flight)
static_assert(kFinOcts % 2 == 0, "the discard loop gives each half-warp one octet");
template <int ACC>
__global__ void __launch_bounds__(kFinThreads) k_bwd_finalize(msa_plan p, const void* dq_pool,
                                                              const float* dk_pool,
                                                              const float* dv_pool,
                                                              __nv_bfloat16* dq,
                                                              __nv_bfloat16* dk,
                                                              __nv_bfloat16* dv) {
  // per warp: kFinOcts octets of [8 heads][128 d] bf16
  __shared__ __align__(16) uint16_t stage[kFinThreads / 32][kFinOcts][8][kHeadDim];
  grid_dep_wait();
  grid_dep_release();
  if (plan_failed(p.header)) return;
  const int lane = threadIdx.x & 31;
  const int64_t n_oct = p.T * (kQHeads / 8);
  const int64_t nk8 = p.T * kKVHeads * kHeadDim / 8;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  uint32_t nonfinite = 0u;  // OR of the exponent fields that were all ones
  if (ACC != MSA_DQ_ACCUM_F32) {
    constexpr bool f16 = ACC == MSA_DQ_ACCUM_F16;
    uint16_t (*st)[8][kHeadDim] = stage[threadIdx.x >> 5];
    const uint4* src = static_cast<const uint4*>(dq_pool);  // [oct][d][8 heads]
    const int64_t nwarps = stride >> 5;
    for (int64_t u = tid >> 5; u * kFinOcts < n_oct; u += nwarps) {
      uint4 w[kFinOcts][4];
#pragma unroll
      for (int o = 0; o < kFinOcts; ++o) {
        const int64_t oct = u * kFinOcts + o;
#pragma unroll
        for (int k = 0; k < 4; ++k)
          w[o][k] = oct < n_oct ? src[oct * kHeadDim + 32 * k + lane] : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int o = 0; o < kFinOcts; ++o) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t ws[4] = {w[o][k].x, w[o][k].y, w[o][k].z, w[o][k].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // heads 2j (low half), 2j + 1 (high half)
            uint32_t b2;
            if (f16) {
              b2 = pack_bf16x2(f16_lo(ws[j]), f16_hi(ws[j]));
              nonfinite |= ((ws[j] & 0x7C00u) == 0x7C00u) |
                           ((ws[j] & 0x7C000000u) == 0x7C000000u);
            } else {
              b2 = ws[j];  // bf16 pool: already the output type
            }
            st[o][2 * j][32 * k + lane] = uint16_t(b2 & 0xFFFFu);
            st[o][2 * j + 1][32 * k + lane] = uint16_t(b2 >> 16);
          }
        }
      }
      __syncwarp();
#pragma unroll
      for (int o = 0; o < kFinOcts; ++o) {
        const int64_t oct = u * kFinOcts + o;
        if (oct < n_oct) {
#pragma unroll
          for (int r = 0; r < 4; ++r) {  // lanes 0-15: head 2r, lanes 16-31: head 2r + 1
            const int h = 2 * r + (lane >> 4);
            const uint4 v = reinterpret_cast<const uint4*>(st[o][h])[lane & 15];
            reinterpret_cast<uint4*>(dq + (oct * 8 + h) * kHeadDim)[lane & 15] = v;
          }
        }
      }
      __syncwarp();
      // the octets' pool lines (16 each) are dead: drop them from L2
#pragma unroll
      for (int o = 0; o < kFinOcts; o += 2) {
        const int64_t oct = u * kFinOcts + o + (lane >> 4);
        if (oct < n_oct) l2_discard_line(src + oct * kHeadDim + 8 * (lane & 15));
      }
    }
  } else {
    const int64_t nq = n_oct * (kHeadDim / 8);
    for (int64_t i = tid; i < nq; i += stride) {
      const int64_t oct = i >> 4;  // token * 8 + head octet
      const int d0 = int(i & 15) * 8;
      uint32_t out[8][4];  // [head in octet][dims pair]
      const float4* src = reinterpret_cast<const float4*>(
          static_cast<const float*>(dq_pool) + (oct * kHeadDim + d0) * 8);
#pragma unroll
      for (int e = 0; e < 8; e += 2) {  // dims d0 + e, d0 + e + 1
        const float4 a0 = src[2 * e], a1 = src[2 * e + 1];
        const float4 b0 = src[2 * e + 2], b1 = src[2 * e + 3];
        const float fa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float fb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int h = 0; h < 8; ++h) out[h][e / 2] = pack_bf16x2(fa[h], fb[h]);
      }
#pragma unroll
      for (int h = 0; h < 8; ++h)
        *reinterpret_cast<uint4*>(dq + (oct * 8 + h) * kHeadDim + d0) =
            make_uint4(out[h][0], out[h][1], out[h][2], out[h][3]);
    }
  }
  // dK / dV: a thread per 128-byte pool line (32 elements), dropped from L2
  // once read
  const int64_t nk32 = nk8 / 4;
  for (int64_t i = tid; i < 2 * nk32; i += stride) {
    const int64_t j = i < nk32 ? i : i - nk32;
    const float4* src = reinterpret_cast<const float4*>(i < nk32 ? dk_pool : dv_pool) + 8 * j;
    float4 a[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) a[e] = src[e];
    uint4* dst = reinterpret_cast<uint4*>(i < nk32 ? dk : dv) + 4 * j;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      dst[e] = make_uint4(pack_bf16x2(a[2 * e].x, a[2 * e].y), pack_bf16x2(a[2 * e].z, a[2 * e].w),
                          pack_bf16x2(a[2 * e + 1].x, a[2 * e + 1].y),
                          pack_bf16x2(a[2 * e + 1].z, a[2 * e + 1].w));
    l2_discard_line(src);
  }
  if (__any_sync(0xffffffffu, nonfinite != 0u) && lane == 0)
    raise_status(p.header, MSA_ERR_RANGE);
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
  void* dq_pool = w + L.off_dq;
  float* dk_pool = reinterpret_cast<float*>(w + L.off_dk);
  float* dv_pool = reinterpret_cast<float*>(w + L.off_dv);

  CUtensorMap mQ, mDO, mK, mV;
  if (make_map_rows(&mQ, q, p.T * kQHeads) != CUDA_SUCCESS ||
      make_map_rows(&mDO, dout, p.T * kQHeads) != CUDA_SUCCESS ||
      make_map_kv(&mK, k, p.T) != CUDA_SUCCESS || make_map_kv(&mV, v, p.T) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;

  const int64_t rows = p.T * kQHeads;
  const int64_t dq_vec = int64_t(dq_elem_bytes(p)) * rows * kHeadDim / 16;
  // dk and dv pools are contiguous in the workspace (dv follows dk)
  const int64_t dkv_vec = int64_t(L.off_dv - L.off_dk) / 16 + p.T * kKVHeads * kHeadDim / 4;
  const int64_t warps = (rows + kDeltaRowsPerWarp - 1) / kDeltaRowsPerWarp;
  // Every kernel may start during its predecessor's tail (launch_k) and
  // waits for it before touching memory; a caller's kernel that never
  // signals counts as signalling when it completes.
  launch_begin("bwd_delta", s);
  cudaError_t e = launch_k(true, k_bwd_delta, dim3(unsigned((warps + 7) / 8)), dim3(256), 0, s, p,
                           static_cast<const __nv_bfloat16*>(o),
                           static_cast<const __nv_bfloat16*>(dout), delta,
                           static_cast<uint4*>(dq_pool), dq_vec,
                           reinterpret_cast<float4*>(dk_pool), dkv_vec);
  launch_end("bwd_delta", s);
  if (e != cudaSuccess) return e;

  static bool attr_set = false;
  if (!attr_set) {
    for (auto fn : {k_bwd_main<MSA_DQ_ACCUM_F16>, k_bwd_main<MSA_DQ_ACCUM_BF16>,
                    k_bwd_main<MSA_DQ_ACCUM_F32>}) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmem);
      if (e != cudaSuccess) return e;
    }
    attr_set = true;
  }
  BwdParams prm{p, lse, delta, dq_pool, dk_pool, dv_pool, scale * kLog2e, scale, p.dq_accum};
  launch_begin("bwd_main", s);
  const unsigned grid = unsigned(device_sm_count());
  auto main_fn = p.dq_accum == MSA_DQ_ACCUM_F32    ? k_bwd_main<MSA_DQ_ACCUM_F32>
                 : p.dq_accum == MSA_DQ_ACCUM_BF16 ? k_bwd_main<MSA_DQ_ACCUM_BF16>
                                                   : k_bwd_main<MSA_DQ_ACCUM_F16>;
  e = launch_k(true, main_fn, dim3(grid), dim3(kBwdThreads), kBwdSmem, s, prm, mQ, mDO, mK, mV);
  launch_end("bwd_main", s);
  if (e != cudaSuccess) return e;
  launch_begin("bwd_finalize", s);
  auto fin_fn = p.dq_accum == MSA_DQ_ACCUM_F32    ? k_bwd_finalize<MSA_DQ_ACCUM_F32>
                : p.dq_accum == MSA_DQ_ACCUM_BF16 ? k_bwd_finalize<MSA_DQ_ACCUM_BF16>
                                                  : k_bwd_finalize<MSA_DQ_ACCUM_F16>;
  e = launch_k(true, fin_fn, dim3(grid * 4), dim3(kFinThreads), 0, s, p, (const void*)dq_pool,
               (const float*)dk_pool, (const float*)dv_pool, static_cast<__nv_bfloat16*>(dq),
               static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv));
  launch_end("bwd_finalize", s);
  return e;
}

}  // namespace msa
