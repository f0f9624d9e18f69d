// plan_static.cu - msa_build_plan_static: the plan builder with its tables in
// device memory that the library itself owns, for callers that cannot
// allocate device memory at the point where they need a plan (for example
// code that runs under a memory manager which forbids allocation, or a
// framework hook that receives only the input buffers).
//
// The scratch is one file-scope __device__ array of kStaticPlanBytes; every
// GPU that loads the library holds it until the process exits.  Host code
// may not use the array's name as a device pointer: its address on the
// current device is looked up with cudaGetSymbolAddress on every call (cheap
// after the first), so a device reset followed by another call still finds
// the live address.
#include "common.cuh"

namespace msa {
msa_status check_device();  // msa_api.cu

namespace {

constexpr size_t kStaticPlanBytes = size_t(16) << 20;  // 16 MiB
__device__ __align__(256) uint8_t g_static_plan[kStaticPlanBytes];

}  // namespace
}  // namespace msa

extern "C" msa_status msa_build_plan_static(const int32_t* q2k, const int32_t* doc_offsets,
                                            int64_t T, int32_t num_docs,
                                            const msa_plan_options* opts, msa_stream_t stream,
                                            msa_plan* out) {
  if (!q2k || !doc_offsets || !out) return MSA_ERR_INVALID_ARG;
  if (T < 1 || T > msa::kMaxTokens || num_docs < 1 || num_docs > T) return MSA_ERR_INVALID_ARG;
  if (msa::plan_layout(T, num_docs).total > msa::kStaticPlanBytes) return MSA_ERR_WORKSPACE;
  const msa_status dev = msa::check_device();
  if (dev != MSA_OK) return dev;
  void* scratch = nullptr;
  if (cudaGetSymbolAddress(&scratch, msa::g_static_plan) != cudaSuccess || !scratch)
    return MSA_ERR_CUDA;
  return msa_build_plan(q2k, doc_offsets, T, num_docs, opts, scratch, msa::kStaticPlanBytes,
                        stream, out);
}
