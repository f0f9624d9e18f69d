// msa_api.cu - the C ABI of libmsa (include/msa.h): argument checks,
// workspace carving, TMA descriptor creation, launch bookkeeping.  No device
// memory is allocated here; every buffer comes from the caller.
#include <atomic>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "common.cuh"

namespace msa {

// ------------------------------------------------------------ launch bookkeeping
namespace {
std::atomic<int64_t> g_launches{0};

struct ProfRec {
  std::string name;
  cudaEvent_t a, b;
  int kernels;
};
struct Prof {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> free_events;
  std::vector<ProfRec> pending;
  std::map<std::string, std::pair<int64_t, double>> acc;
  std::map<cudaStream_t, cudaEvent_t> open;  // begin event per stream
};
Prof& prof() {
  static Prof p;
  return p;
}
cudaEvent_t take_event(Prof& p) {
  if (!p.free_events.empty()) {
    cudaEvent_t e = p.free_events.back();
    p.free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}
// Fold finished records into the totals (caller holds the lock).
void drain(Prof& p, bool wait) {
  std::vector<ProfRec> keep;
  for (auto& r : p.pending) {
    if (wait) cudaEventSynchronize(r.b);
    if (cudaEventQuery(r.b) == cudaSuccess) {
      float ms = 0.f;
      cudaEventElapsedTime(&ms, r.a, r.b);
      auto& slot = p.acc[r.name];
      slot.first += r.kernels;
      slot.second += ms;
      p.free_events.push_back(r.a);
      p.free_events.push_back(r.b);
    } else {
      keep.push_back(r);
    }
  }
  p.pending.swap(keep);
}
}  // namespace

bool profiling_on() { return prof().on; }

void launch_begin(const char* name, cudaStream_t s) {
  (void)name;
  Prof& p = prof();
  if (!p.on) return;
  std::lock_guard<std::mutex> g(p.mu);
  cudaEvent_t a = take_event(p);
  cudaEventRecord(a, s);
  p.open[s] = a;
}

void launch_end(const char* name, cudaStream_t s, int kernels) {
  g_launches.fetch_add(kernels);
  Prof& p = prof();
  if (!p.on) return;
  std::lock_guard<std::mutex> g(p.mu);
  auto it = p.open.find(s);
  if (it == p.open.end()) return;
  cudaEvent_t b = take_event(p);
  cudaEventRecord(b, s);
  p.pending.push_back(ProfRec{name, it->second, b, kernels});
  p.open.erase(it);
  if (p.pending.size() > 4096) drain(p, false);
}

// ------------------------------------------------------------ device helpers
int device_sm_count() {
  int dev = 0;
  cudaGetDevice(&dev);
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> g(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  cache[dev] = n;
  return n;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}


bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
}  // namespace

// The library runs on sm_100 / sm_103 class devices only (also used by
// plan_static.cu).
msa_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MSA_ERR_CUDA;
  int major = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return MSA_ERR_CUDA;
  return major == 10 ? MSA_OK : MSA_ERR_UNSUPPORTED;
}

// [rows, 128] bf16 rows (Q or dO viewed as [T*64, 128]); box = 16 rows x 64
// columns, 128-byte swizzle: one box is the 16 heads of one index head of
// one token, half of the head dimension.
CUresult make_map_rows(CUtensorMap* m, const void* base, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t gd[2] = {cuuint64_t(kHeadDim), cuuint64_t(rows)};
  cuuint64_t gs[1] = {cuuint64_t(kHeadDim * 2)};
  cuuint32_t box[2] = {64, 16};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gd, gs, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// [T, 4, 128] bf16 (K or V); box = 128 tokens of one KV head x 64 columns.
// Rows past T read as zero.
CUresult make_map_kv(CUtensorMap* m, const void* base, int64_t T) {
  auto fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t gd[3] = {cuuint64_t(kHeadDim), cuuint64_t(kKVHeads), cuuint64_t(T)};
  cuuint64_t gs[2] = {cuuint64_t(kHeadDim * 2), cuuint64_t(kKVHeads * kHeadDim * 2)};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gd, gs, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// [rows, 128] fp32 pool (forward O accumulation) as the destination of bulk
// tensor reductions; box = 16 rows x 32 columns (128 bytes), 128-byte swizzle,
// so a tile row staged by one thread is spread over all shared-memory banks.
CUresult make_map_pool32(CUtensorMap* m, const void* base, int64_t rows) {
  auto fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_FOUND;
  cuuint64_t gd[2] = {cuuint64_t(kHeadDim), cuuint64_t(rows)};
  cuuint64_t gs[1] = {cuuint64_t(kHeadDim * 4)};
  cuuint32_t box[2] = {32, 16};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), gd, gs, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace msa

using namespace msa;

#ifdef MSA_TEST_STARVE
namespace msa {
cudaError_t test_set_starve_fwd(int which);  // attn_fwd.cu
cudaError_t test_set_starve_bwd(int which);  // attn_bwd.cu
}  // namespace msa
// Test-only build: make CTA 0 of one kernel (1: fwd_group, 2: fwd_main,
// 3: bwd_main, 0: none) leave out its first Q tile, so that a bounded
// pipeline wait runs out and the call reports MSA_ERR_TIMEOUT.
extern "C" msa_status msa_test_starve(int32_t which) {
  if (which < 0 || which > 3) return MSA_ERR_INVALID_ARG;
  if (test_set_starve_fwd(which) != cudaSuccess || test_set_starve_bwd(which) != cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}
#endif

// ------------------------------------------------------------ C ABI
extern "C" {

const char* msa_status_string(msa_status s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED";
    case MSA_ERR_ALIGNMENT: return "MSA_ERR_ALIGNMENT";
    case MSA_ERR_WORKSPACE: return "MSA_ERR_WORKSPACE";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA";
    case MSA_ERR_BAD_Q2K: return "MSA_ERR_BAD_Q2K";
    case MSA_ERR_BAD_OFFSETS: return "MSA_ERR_BAD_OFFSETS";
    case MSA_ERR_TIMEOUT: return "MSA_ERR_TIMEOUT";
    case MSA_ERR_CAPACITY: return "MSA_ERR_CAPACITY";
    case MSA_ERR_RANGE: return "MSA_ERR_RANGE";
  }
  return "MSA_ERR_UNKNOWN";
}

msa_status msa_plan_workspace_bytes(int64_t T, int32_t num_docs, size_t* bytes) {
  if (!bytes || T < 1 || T > kMaxTokens || num_docs < 1 || num_docs > T) return MSA_ERR_INVALID_ARG;
  *bytes = plan_layout(T, num_docs).total;
  return MSA_OK;
}

msa_status msa_build_plan(const int32_t* q2k, const int32_t* doc_offsets, int64_t T,
                          int32_t num_docs, const msa_plan_options* opts, void* workspace,
                          size_t workspace_bytes, msa_stream_t stream, msa_plan* out) {
  if (!q2k || !doc_offsets || !workspace || !out) return MSA_ERR_INVALID_ARG;
  if (T < 1 || T > kMaxTokens || num_docs < 1 || num_docs > T) return MSA_ERR_INVALID_ARG;
  const int32_t Z = opts ? opts->super_block : 64;
  const int32_t acc = opts ? opts->dq_accum : MSA_DQ_ACCUM_F16;
  const int32_t oacc = opts ? opts->o_accum : MSA_O_ACCUM_F32;
  const int32_t dense = opts ? opts->dense_blocks : 0;
  if (Z < 0 || acc < MSA_DQ_ACCUM_F16 || acc > MSA_DQ_ACCUM_F32) return MSA_ERR_INVALID_ARG;
  if (dense < -1 || dense > kMaxDenseBlocks) return MSA_ERR_INVALID_ARG;
  if (oacc != MSA_O_ACCUM_F32 && oacc != MSA_O_ACCUM_BF16) return MSA_ERR_INVALID_ARG;
  // A bf16 O pool rounds every partial sum to 8 bits and O once more on the
  // store: up to one bf16 ulp of O (2^-6 for |O| in [2, 4)), above the 1e-2
  // max-abs bar the forward is held to.  Not offered.
  if (oacc == MSA_O_ACCUM_BF16) return MSA_ERR_UNSUPPORTED;
  if (!aligned16(q2k) || !aligned16(workspace) || (reinterpret_cast<uintptr_t>(doc_offsets) & 3u))
    return MSA_ERR_ALIGNMENT;
  const PlanLayout L = plan_layout(T, num_docs);
  if (workspace_bytes < L.total) return MSA_ERR_WORKSPACE;
  const msa_status dev = check_device();
  if (dev != MSA_OK) return dev;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  msa_plan p{};
  p.T = T;
  p.num_docs = num_docs;
  p.super_block = Z;
  p.dq_accum = acc;
  p.o_accum = oacc;
  p.dense_blocks = dense == 0 ? kDefaultDenseBlocks : (dense < 0 ? 0 : dense);
  p.nb_cap = L.nb_cap;
  p.tri_cap = L.tri_cap;
  p.nnz_cap = L.nnz_cap;
  p.task_cap = L.task_cap;
  p.q2k = q2k;
  p.doc_offsets = doc_offsets;
  p.header = reinterpret_cast<int64_t*>(w + L.off_header);
  p.doc_info = reinterpret_cast<int32_t*>(w + L.off_doc_info);
  p.doc_tri = reinterpret_cast<int64_t*>(w + L.off_doc_tri);
  p.cnt = reinterpret_cast<int32_t*>(w + L.off_cnt);
  p.off = reinterpret_cast<int32_t*>(w + L.off_off);
  p.col = reinterpret_cast<int32_t*>(w + L.off_col);
  p.tcnt = reinterpret_cast<int32_t*>(w + L.off_tcnt);
  p.toff = reinterpret_cast<int32_t*>(w + L.off_toff);
  p.tasks = reinterpret_cast<int32_t*>(w + L.off_tasks);
  p.scan_tmp = reinterpret_cast<int32_t*>(w + L.off_scan);
  p.scan_tmp_len = L.scan_tmp_len;
  p.item_cap = L.item_cap;
  p.grouped = reinterpret_cast<uint8_t*>(w + L.off_grouped);
  p.items = reinterpret_cast<int32_t*>(w + L.off_items);
  p.fflag = reinterpret_cast<int32_t*>(w + L.off_fflag);
  p.fpos = reinterpret_cast<int32_t*>(w + L.off_fpos);
  p.ftasks = reinterpret_cast<int32_t*>(w + L.off_ftasks);
  p.rows = reinterpret_cast<int32_t*>(w + L.off_rows);
  if (launch_plan(p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MSA_ERR_CUDA;
  *out = p;
  return MSA_OK;
}

static msa_status check_plan(const msa_plan* plan) {
  if (!plan || plan->T < 1 || !plan->header || !plan->tasks || !plan->ftasks || !plan->items ||
      !plan->grouped || !plan->rows)
    return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

msa_status msa_forward_workspace_bytes(const msa_plan* plan, size_t* bytes) {
  if (check_plan(plan) != MSA_OK || !bytes) return MSA_ERR_INVALID_ARG;
  *bytes = forward_workspace_bytes(*plan);
  return MSA_OK;
}

msa_status msa_backward_workspace_bytes(const msa_plan* plan, size_t* bytes) {
  if (check_plan(plan) != MSA_OK || !bytes) return MSA_ERR_INVALID_ARG;
  *bytes = backward_workspace_bytes(*plan);
  return MSA_OK;
}

msa_status msa_forward(const msa_plan* plan, const void* q, const void* k, const void* v,
                       float softmax_scale, void* o, float* lse, void* workspace,
                       size_t workspace_bytes, msa_stream_t stream) {
  if (check_plan(plan) != MSA_OK || !q || !k || !v || !o || !lse || !workspace)
    return MSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale > 1e30f) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(workspace))
    return MSA_ERR_ALIGNMENT;
  if (workspace_bytes < forward_workspace_bytes(*plan)) return MSA_ERR_WORKSPACE;
  const msa_status dev = check_device();
  if (dev != MSA_OK) return dev;
  if (launch_forward(*plan, q, k, v, softmax_scale, o, lse, workspace,
                     reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}

msa_status msa_backward(const msa_plan* plan, const void* q, const void* k, const void* v,
                        const void* o, const float* lse, const void* dout, float softmax_scale,
                        void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                        msa_stream_t stream) {
  if (check_plan(plan) != MSA_OK || !q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv ||
      !workspace)
    return MSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.f) || softmax_scale > 1e30f) return MSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv) ||
      !aligned16(workspace))
    return MSA_ERR_ALIGNMENT;
  if (workspace_bytes < backward_workspace_bytes(*plan)) return MSA_ERR_WORKSPACE;
  const msa_status dev = check_device();
  if (dev != MSA_OK) return dev;
  if (launch_backward(*plan, q, k, v, o, lse, dout, softmax_scale, dq, dk, dv, workspace,
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}

msa_status msa_read_status(const msa_plan* plan, msa_stream_t stream) {
  if (check_plan(plan) != MSA_OK) return MSA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MSA_ERR_CUDA;
  int64_t bits = 0;
  if (cudaMemcpy(&bits, plan->header + kHdrStatus, sizeof bits, cudaMemcpyDeviceToHost) !=
      cudaSuccess)
    return MSA_ERR_CUDA;
  for (int c = 1; c < 63; ++c)
    if (bits & (int64_t(1) << c)) return static_cast<msa_status>(c);
  return MSA_OK;
}

msa_status msa_plan_counts(const msa_plan* plan, msa_stream_t stream, int64_t* counts) {
  if (check_plan(plan) != MSA_OK || !counts) return MSA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MSA_ERR_CUDA;
  int64_t h[kHdrWords];
  if (cudaMemcpy(h, plan->header, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MSA_ERR_CUDA;
  counts[0] = h[kHdrNB];
  counts[1] = h[kHdrNnz];
  counts[2] = h[kHdrTasks];
  counts[3] = h[kHdrPairs];
  counts[4] = h[kHdrTri];
  counts[5] = h[kHdrItems];
  counts[6] = h[kHdrFTasks];
  return MSA_OK;
}

msa_status msa_plan_export(const msa_plan* plan, msa_stream_t stream, int32_t* col,
                           int64_t col_capacity, int32_t* tasks, int64_t task_capacity) {
  int64_t c[7];
  msa_status st = msa_plan_counts(plan, stream, c);
  if (st != MSA_OK) return st;
  if ((col && col_capacity < c[1]) || (tasks && task_capacity < c[2])) return MSA_ERR_INVALID_ARG;
  if (col && c[1] > 0 &&
      cudaMemcpy(col, plan->col, sizeof(int32_t) * c[1], cudaMemcpyDeviceToHost) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (tasks && c[2] > 0 &&
      cudaMemcpy(tasks, plan->tasks, sizeof(int32_t) * 4 * c[2], cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}

msa_status msa_plan_export_groups(const msa_plan* plan, msa_stream_t stream, uint8_t* grouped,
                                  int64_t grouped_capacity, int32_t* items,
                                  int64_t item_capacity, int32_t* ftasks,
                                  int64_t ftask_capacity) {
  int64_t c[7];
  msa_status st = msa_plan_counts(plan, stream, c);
  if (st != MSA_OK) return st;
  if ((grouped && grouped_capacity < plan->T) || (items && item_capacity < c[5]) ||
      (ftasks && ftask_capacity < c[6]))
    return MSA_ERR_INVALID_ARG;
  if (grouped && cudaMemcpy(grouped, plan->grouped, size_t(kKVHeads) * plan->T,
                            cudaMemcpyDeviceToHost) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (items && c[5] > 0 &&
      cudaMemcpy(items, plan->items, sizeof(int32_t) * kItemWords * c[5],
                 cudaMemcpyDeviceToHost) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (ftasks && c[6] > 0 &&
      cudaMemcpy(ftasks, plan->ftasks, sizeof(int32_t) * 4 * c[6], cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return MSA_ERR_CUDA;
  return MSA_OK;
}

msa_status msa_profile_enable(int32_t on) {
  Prof& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  p.on = on != 0;
  return MSA_OK;
}

msa_status msa_profile_reset(void) {
  Prof& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  drain(p, true);
  p.acc.clear();
  return MSA_OK;
}

msa_status msa_profile_read(const char* name, int64_t* launches, double* total_ms) {
  if (!name || !launches || !total_ms) return MSA_ERR_INVALID_ARG;
  Prof& p = prof();
  std::lock_guard<std::mutex> g(p.mu);
  drain(p, true);
  auto it = p.acc.find(name);
  *launches = it == p.acc.end() ? 0 : it->second.first;
  *total_ms = it == p.acc.end() ? 0.0 : it->second.second;
  return MSA_OK;
}

int64_t msa_launch_count(void) { return g_launches.load(); }

}  // extern "C"
