// plan_static.cu - msa_build_plan_static: the plan builder with its tables in
// device memory that the library itself owns, for callers that cannot
// allocate device memory at the point where they need a plan (for example
// code that runs under a memory manager which forbids allocation, or a
// framework hook that receives only the input buffers).
//
// The scratch is one file-scope __device__ array of kStaticPlanBytes; every
// GPU that loads the library holds it until the process exits.  Its address
// is looked up once per device with cudaGetSymbolAddress (host code may not
// use the array's name as a device pointer).
#include <map>
#include <mutex>

#include "common.cuh"

namespace msa {
namespace {

constexpr size_t kStaticPlanBytes = size_t(16) << 20;  // 16 MiB
__device__ __align__(256) uint8_t g_static_plan[kStaticPlanBytes];

std::mutex g_static_mu;
std::map<int, void*> g_static_addr;  // device ordinal -> device address of g_static_plan

// Device address of the scratch array on the current device (looked up on
// the first call per device).  Returns nullptr if the lookup fails.
void* static_plan_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> g(g_static_mu);
  auto it = g_static_addr.find(dev);
  if (it != g_static_addr.end()) return it->second;
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_static_plan) != cudaSuccess || ptr == nullptr) {
    cudaGetLastError();  // clear the error so later runtime calls do not report it
    return nullptr;
  }
  g_static_addr[dev] = ptr;
  return ptr;
}

}  // namespace
}  // namespace msa

extern "C" msa_status msa_build_plan_static(const int32_t* q2k, const int32_t* doc_offsets,
                                            int64_t T, int32_t num_docs,
                                            const msa_plan_options* opts, msa_stream_t stream,
                                            msa_plan* out) {
  if (!q2k || !doc_offsets || !out) return MSA_ERR_INVALID_ARG;
  if (T < 1 || T > msa::kMaxTokens || num_docs < 1 || num_docs > T) return MSA_ERR_INVALID_ARG;
  if (msa::plan_layout(T, num_docs).total > msa::kStaticPlanBytes) return MSA_ERR_WORKSPACE;
  void* scratch = msa::static_plan_scratch();
  if (!scratch) return MSA_ERR_CUDA;
  return msa_build_plan(q2k, doc_offsets, T, num_docs, opts, scratch, msa::kStaticPlanBytes,
                        stream, out);
}
