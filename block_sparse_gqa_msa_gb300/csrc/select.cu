// select.cu - the index scorer and top-16 block selection that produce q2k.
//
// The pages name the step (an indexer scores the key blocks of each query's
// document and the query keeps the best 16) without a scoring formula.  The
// plainest reading, stated in include/msa.h: a block's summary is the mean of
// its index keys, a query's score for a block is the dot product of its index
// query with that summary; blocks 0 .. b (b = the query's own block) are the
// candidates, all of them when there are at most 16, else the 16 best by
// (score descending, block ascending), optionally always keeping block 0 and
// block b.  Scores are fp32 with a fixed order of operations (the block sum
// key by key then divided by the key count, the dot product channel by
// channel with fused multiply-adds), so the ranking is reproducible.
//
// Kernels:
//   sel_summary  one CTA per 128-token window: the block summaries of the
//                document blocks that start in it (thread = index head x channel)
//   sel_topk     one warp per (token, index head): scores of the candidate
//                blocks, a lane-local best-K (K = the lane's candidate count
//                rounded up to 2, 4, 8 or 16) kept with a replace-the-worst
//                rule, then 16 rounds of warp-wide selection
#include <cfloat>
#include <climits>

#include "common.cuh"

namespace msa {
namespace {

constexpr int kSelWarps = 8;

__device__ __forceinline__ int32_t sel_doc_of(const int32_t* offs, int32_t D, int64_t t) {
  int32_t lo = 0, hi = D - 1;  // largest d with offs[d] <= t
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (offs[mid] <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}
// Summary row of document block v: floor(o_d / 128) + d + v is unique over
// all (d, v) and below T / 128 + D + 1.
__device__ __forceinline__ int64_t sel_slot(int32_t od, int32_t d, int32_t v) {
  return int64_t(od >> 7) + d + v;
}
// (s1, v1) ranks before (s2, v2)?
__device__ __forceinline__ bool sel_better(float s1, int32_t v1, float s2, int32_t v2) {
  return s1 > s2 || (s1 == s2 && v1 < v2);
}

__global__ void __launch_bounds__(512) k_sel_summary(const __nv_bfloat16* __restrict__ ik,
                                                     int64_t T, int32_t dim,
                                                     const int32_t* __restrict__ offs, int32_t D,
                                                     float* __restrict__ summ, int64_t slots) {
  __shared__ int32_t starts[128];
  __shared__ int nstart;
  if (threadIdx.x == 0) nstart = 0;
  __syncthreads();
  const int64_t t0 = int64_t(blockIdx.x) * 128;
  if (threadIdx.x < 128 && t0 + threadIdx.x < T) {
    const int64_t t = t0 + threadIdx.x;
    const int32_t d = sel_doc_of(offs, D, t);
    if (((t - offs[d]) & 127) == 0) starts[atomicAdd(&nstart, 1)] = int32_t(t);
  }
  __syncthreads();
  const int g = int(threadIdx.x) / dim, c = int(threadIdx.x) % dim;
  if (g >= kKVHeads) return;
  for (int i = 0; i < nstart; ++i) {
    const int32_t t = starts[i];
    const int32_t d = sel_doc_of(offs, D, t);
    const int32_t v = (t - offs[d]) >> 7;
    const int32_t n = min(128, offs[d + 1] - t);
    const int64_t slot = sel_slot(offs[d], d, v);
    if (n <= 0 || slot < 0 || slot >= slots) continue;
    float acc = 0.f;
    const __nv_bfloat16* col = ik + (int64_t(t) * kKVHeads + g) * dim + c;
#pragma unroll 8
    for (int32_t j = 0; j < n; ++j) acc += __bfloat162float(col[int64_t(j) * kKVHeads * dim]);
    summ[(int64_t(g) * slots + slot) * dim + c] = __fdiv_rn(acc, float(n));
  }
}

// The selection of one (token, index head) by one warp.  Each lane keeps its
// best K candidates (K >= the lane's candidate count, or 16); `need` rounds
// of warp-wide best-of-the-rest then pick the winners into chosen[0..need).
template <int K>
__device__ __forceinline__ void select_row(const float* rows, const float* q, int32_t dim,
                                           int32_t lo, int32_t hi, int need, int lane,
                                           int32_t* chosen) {
  float ks[K];
  int32_t kv[K];
#pragma unroll
  for (int k = 0; k < K; ++k) {
    ks[k] = -FLT_MAX;
    kv[k] = INT_MAX;
  }
  int worst = 0;  // the kept entry every other one ranks before
  for (int32_t v = lo + lane; v <= hi; v += 32) {
    const float4* r4 = reinterpret_cast<const float4*>(rows + int64_t(v) * dim);
    float acc = 0.f;
    for (int c4 = 0; c4 < dim / 4; ++c4) {
      const float4 s = r4[c4];
      acc = fmaf(q[4 * c4 + 0], s.x, acc);
      acc = fmaf(q[4 * c4 + 1], s.y, acc);
      acc = fmaf(q[4 * c4 + 2], s.z, acc);
      acc = fmaf(q[4 * c4 + 3], s.w, acc);
    }
    float ws = -FLT_MAX;
    int32_t wv = INT_MAX;
#pragma unroll
    for (int k = 0; k < K; ++k)
      if (k == worst) { ws = ks[k]; wv = kv[k]; }
    if (sel_better(acc, v, ws, wv)) {
#pragma unroll
      for (int k = 0; k < K; ++k)
        if (k == worst) { ks[k] = acc; kv[k] = v; }
      worst = 0;
      float bs = ks[0];
      int32_t bv = kv[0];
#pragma unroll
      for (int k = 1; k < K; ++k)
        if (sel_better(bs, bv, ks[k], kv[k])) { worst = k; bs = ks[k]; bv = kv[k]; }
    }
  }
  for (int r = 0; r < need; ++r) {
    float bs = -FLT_MAX;
    int32_t bv = INT_MAX;
#pragma unroll
    for (int k = 0; k < K; ++k)
      if (sel_better(ks[k], kv[k], bs, bv)) { bs = ks[k]; bv = kv[k]; }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float os = __shfl_xor_sync(0xffffffffu, bs, o);
      const int32_t ov = __shfl_xor_sync(0xffffffffu, bv, o);
      if (sel_better(os, ov, bs, bv)) { bs = os; bv = ov; }
    }
#pragma unroll
    for (int k = 0; k < K; ++k)
      if (kv[k] == bv) { ks[k] = -FLT_MAX; kv[k] = INT_MAX; }
    if (lane == 0) chosen[r] = bv;
  }
}

__global__ void __launch_bounds__(kSelWarps * 32) k_sel_topk(
    const __nv_bfloat16* __restrict__ iq, const float* __restrict__ summ, int64_t slots,
    int64_t T, int32_t dim, const int32_t* __restrict__ offs, int32_t D, int32_t force_local,
    int32_t* __restrict__ q2k) {
  __shared__ float sq[kSelWarps][128];
  __shared__ int32_t chosen[kSelWarps][kTopK];
  const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
  const int64_t nwarps = int64_t(gridDim.x) * kSelWarps;
  for (int64_t w = int64_t(blockIdx.x) * kSelWarps + wl; w < 4 * T; w += nwarps) {
    const int64_t t = w >> 2;
    const int g = int(w & 3);
    int32_t* out = q2k + (int64_t(g) * T + t) * kTopK;
    const int32_t d = sel_doc_of(offs, D, t);
    const int32_t s0 = offs[d];
    const int32_t b = int32_t((t - s0) >> 7);
    const int64_t row0 = sel_slot(s0, d, 0);
    if (b + 1 <= kTopK || row0 < 0 || row0 + b >= slots) {
      if (lane < kTopK) out[lane] = lane <= b && b + 1 <= kTopK ? lane : -1;
      continue;
    }
    for (int c = lane; c < dim; c += 32) sq[wl][c] = __bfloat162float(iq[(t * kKVHeads + g) * dim + c]);
    __syncwarp();
    const float* rows = summ + (int64_t(g) * slots + row0) * dim;
    const int32_t lo = force_local ? 1 : 0, hi = force_local ? b - 1 : b;
    const int need = force_local ? kTopK - 2 : kTopK;
    const int32_t per_lane = (hi - lo + 32) / 32;  // candidates per lane, rounded up
    if (per_lane <= 2)
      select_row<2>(rows, sq[wl], dim, lo, hi, need, lane, chosen[wl]);
    else if (per_lane <= 4)
      select_row<4>(rows, sq[wl], dim, lo, hi, need, lane, chosen[wl]);
    else if (per_lane <= 8)
      select_row<8>(rows, sq[wl], dim, lo, hi, need, lane, chosen[wl]);
    else
      select_row<kTopK>(rows, sq[wl], dim, lo, hi, need, lane, chosen[wl]);
    if (force_local && lane == 0) {
      chosen[wl][kTopK - 2] = 0;
      chosen[wl][kTopK - 1] = b;
    }
    __syncwarp();
    if (lane < kTopK) {  // ascending order: each value's rank among the 16 distinct values
      const int32_t mine = chosen[wl][lane];
      int rank = 0;
#pragma unroll
      for (int k = 0; k < kTopK; ++k) rank += chosen[wl][k] < mine ? 1 : 0;
      out[rank] = mine;
    }
    __syncwarp();
  }
}

}  // namespace

int device_sm_count();

int64_t select_slots(int64_t T, int32_t num_docs) { return T / 128 + num_docs + 1; }

cudaError_t launch_select(const void* iq, const void* ik, int64_t T, int32_t dim,
                          const int32_t* offs, int32_t D, int32_t force_local, int32_t* q2k,
                          void* ws, cudaStream_t s) {
  const int64_t slots = select_slots(T, D);
  float* summ = static_cast<float*>(ws);
  launch_begin("sel_summary", s);
  k_sel_summary<<<unsigned((T + 127) / 128), unsigned(4 * dim), 0, s>>>(
      static_cast<const __nv_bfloat16*>(ik), T, dim, offs, D, summ, slots);
  launch_end("sel_summary", s);
  launch_begin("sel_topk", s);
  k_sel_topk<<<unsigned(device_sm_count() * 8), kSelWarps * 32, 0, s>>>(
      static_cast<const __nv_bfloat16*>(iq), summ, slots, T, dim, offs, D, force_local, q2k);
  launch_end("sel_topk", s);
  return cudaGetLastError();
}

}  // namespace msa

extern "C" msa_status msa_select_workspace_bytes(int64_t T, int32_t num_docs, int32_t dim,
                                                 size_t* bytes) {
  if (!bytes || T < 1 || T > msa::kMaxTokens || num_docs < 1 || num_docs > T || dim < 8 ||
      dim > 128 || dim % 8)
    return MSA_ERR_INVALID_ARG;
  *bytes = size_t(4) * size_t(msa::select_slots(T, num_docs)) * size_t(dim) * sizeof(float);
  return MSA_OK;
}

extern "C" msa_status msa_select_blocks(const void* iq, const void* ik, int64_t T, int32_t dim,
                                        const int32_t* doc_offsets, int32_t num_docs,
                                        int32_t force_local, int32_t* q2k, void* workspace,
                                        size_t workspace_bytes, msa_stream_t stream) {
  size_t need = 0;
  if (!iq || !ik || !doc_offsets || !q2k || !workspace) return MSA_ERR_INVALID_ARG;
  if (msa_select_workspace_bytes(T, num_docs, dim, &need) != MSA_OK) return MSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(iq) | reinterpret_cast<uintptr_t>(ik) |
       reinterpret_cast<uintptr_t>(workspace)) & 15)
    return MSA_ERR_ALIGNMENT;
  if (workspace_bytes < need) return MSA_ERR_WORKSPACE;
  const cudaError_t e = msa::launch_select(iq, ik, T, dim, doc_offsets, num_docs,
                                           force_local ? 1 : 0, q2k, workspace,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}
