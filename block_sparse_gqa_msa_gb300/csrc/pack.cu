// pack.cu - padded packed rows [B][S][row] <-> compact THD [T][row].
//
// Both directions are streaming copies of 16-byte vectors (HBM-bound: the
// bytes moved are the roofline).  A warp copies one token row at a time; the
// row's place in the compact layout comes from an exclusive prefix sum of
// the row lengths computed on the device first.
#include "common.cuh"

namespace msa {
namespace {

// Exclusive prefix sum of the clamped row lengths: offsets[0..B].  One CTA.
__global__ void __launch_bounds__(1024) k_row_offsets(const int32_t* row_len, int32_t B,
                                                      int32_t S, int32_t* offsets) {
  __shared__ int32_t warp_tot[32];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int32_t base = 0; base < B; base += blockDim.x) {
    const int32_t i = base + threadIdx.x;
    const int32_t len = i < B ? min(max(row_len[i], 0), S) : 0;
    int32_t x = len;  // inclusive scan within the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int32_t w = lane < int(blockDim.x >> 5) ? warp_tot[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_tot[lane] = w;  // inclusive scan of warp totals
    }
    __syncthreads();
    const int32_t before = carry + (warp > 0 ? warp_tot[warp - 1] : 0);
    if (i < B) offsets[i] = before + x - len;
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) carry = before + x;
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[B] = carry;
}

// One warp per token row (b, s), its lanes over the row's 16-byte vectors.
template <bool kPack>
__global__ void __launch_bounds__(256) k_pack(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                              int32_t B, int32_t S, int32_t vecs,
                                              const int32_t* __restrict__ row_len,
                                              const int32_t* __restrict__ offsets) {
  const int lane = threadIdx.x & 31;
  const int64_t tokens = int64_t(B) * S;
  const int64_t wstride = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t tok = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; tok < tokens;
       tok += wstride) {
    const int32_t b = int32_t(tok / S), s = int32_t(tok - int64_t(b) * S);
    const int32_t len = min(max(row_len[b], 0), S);
    const int64_t y_row = int64_t(offsets[b]) + s;
    const uint4* sp = src + (kPack ? tok : y_row) * vecs;
    uint4* dp = dst + (kPack ? y_row : tok) * vecs;
    if (s < len) {
      for (int32_t e = lane; e < vecs; e += 32) dp[e] = sp[e];
    } else if (!kPack) {
      for (int32_t e = lane; e < vecs; e += 32) dp[e] = make_uint4(0, 0, 0, 0);
    }
  }
}

}  // namespace

int device_sm_count();

cudaError_t launch_pack(const void* x, int32_t B, int32_t S, int32_t row_bytes,
                        const int32_t* row_len, void* y, int32_t* row_offsets, cudaStream_t s) {
  launch_begin("pack_offsets", s);
  k_row_offsets<<<1, 1024, 0, s>>>(row_len, B, S, row_offsets);
  launch_end("pack_offsets", s);
  launch_begin("pack_thd", s);
  k_pack<true><<<unsigned(device_sm_count() * 8), 256, 0, s>>>(
      static_cast<const uint4*>(x), static_cast<uint4*>(y), B, S, row_bytes / 16, row_len,
      row_offsets);
  launch_end("pack_thd", s);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const void* y, int32_t B, int32_t S, int32_t row_bytes,
                          const int32_t* row_len, const int32_t* row_offsets, void* x,
                          cudaStream_t s) {
  launch_begin("unpack_bshd", s);
  k_pack<false><<<unsigned(device_sm_count() * 8), 256, 0, s>>>(
      static_cast<const uint4*>(y), static_cast<uint4*>(x), B, S, row_bytes / 16, row_len,
      row_offsets);
  launch_end("unpack_bshd", s);
  return cudaGetLastError();
}

}  // namespace msa

extern "C" msa_status msa_pack_thd(const void* x, int32_t B, int32_t S, int32_t row_bytes,
                                   const int32_t* row_len, void* y, int32_t* row_offsets,
                                   msa_stream_t stream) {
  if (!x || !row_len || !y || !row_offsets) return MSA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || row_bytes < 16 || row_bytes % 16 || int64_t(B) * S >= (int64_t(1) << 31))
    return MSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) return MSA_ERR_ALIGNMENT;
  const cudaError_t e = msa::launch_pack(x, B, S, row_bytes, row_len, y, row_offsets,
                                         static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

extern "C" msa_status msa_unpack_bshd(const void* y, int32_t B, int32_t S, int32_t row_bytes,
                                      const int32_t* row_len, const int32_t* row_offsets,
                                      void* x, msa_stream_t stream) {
  if (!x || !row_len || !y || !row_offsets) return MSA_ERR_INVALID_ARG;
  if (B < 1 || S < 1 || row_bytes < 16 || row_bytes % 16 || int64_t(B) * S >= (int64_t(1) << 31))
    return MSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) return MSA_ERR_ALIGNMENT;
  const cudaError_t e = msa::launch_unpack(y, B, S, row_bytes, row_len, row_offsets, x,
                                           static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}
