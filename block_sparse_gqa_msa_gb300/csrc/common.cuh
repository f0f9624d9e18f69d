// common.cuh - shapes, plan layout and status bits shared by the MSA kernels.
//
// Fixed topology of the method (NeMo-Automodel PR "feat(minimax-m3): add SM100
// MSA sparse attention with custom backward", section "Supported scope"):
// 64 query heads, 4 KV heads, 4 index heads, head dim 128, key block 128,
// top-16 selection.  Query head h reads KV / index head h / 16.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include "../../include/msa.h"

namespace msa {

constexpr int kQHeads = 64;
constexpr int kKVHeads = 4;
constexpr int kHeadsPerGroup = 16;  // query heads per index head
constexpr int kHeadDim = 128;
constexpr int kBlock = 128;         // keys per block
constexpr int kTopK = 16;           // q2k slots
constexpr int kTaskQueries = 8;     // queries per task: 8 x 16 heads = 128 rows
constexpr int kMaxTokens = 1 << 20;

// Header slots (int64) in the plan workspace.
enum HeaderSlot {
  kHdrStatus = 0,   // OR of (1 << msa_status) for device-detected errors
  kHdrNB = 1,       // number of 128-key blocks over all documents
  kHdrTri = 2,      // count entries: 4 * sum_d nblk_d (nblk_d + 1) / 2
  kHdrNnz = 3,      // CSR entries
  kHdrTasks = 4,    // tasks
  kHdrPairs = 5,    // attended (query, head, key) triples
  kHdrTriPerG = 6,  // count entries per index head
  kHdrItems = 7,    // octet-group items of the forward
  kHdrFTasks = 8,   // tasks of the forward's pooled task list
  kHdrRows = 9,     // (token, index head) pairs outside the octet groups
  kHdrCost = 16,    // [kHdrCost + c]: items of cost c (1..128)
  kHdrCostFill = 145,  // placement counters of the items, per cost
  kHdrWords = 288
};
constexpr int kMaxDenseBlocks = 64;   // a dense octet's token masks are 64-bit words
constexpr int kDefaultDenseBlocks = 32;
constexpr int kMaxItemCost = 2 * kMaxDenseBlocks;  // an item: at most 2 octets x 64 blocks

__device__ __forceinline__ void raise_status(int64_t* header, msa_status s) {
  atomicOr(reinterpret_cast<unsigned long long*>(header + kHdrStatus),
           1ull << static_cast<int>(s));
}
// Status bits that are warnings about one call's result, not plan failures.
constexpr int64_t kStatusWarnings = int64_t(1) << MSA_ERR_RANGE;
__device__ __forceinline__ bool plan_failed(const int64_t* header) {
  return (*reinterpret_cast<const volatile int64_t*>(header + kHdrStatus) & ~kStatusWarnings) != 0;
}
__device__ __forceinline__ void clear_warnings(int64_t* header) {
  atomicAnd(reinterpret_cast<unsigned long long*>(header + kHdrStatus),
            ~static_cast<unsigned long long>(kStatusWarnings));
}

// Per-document record in the plan: start token, length, blocks, first global block.
struct DocInfo {
  int32_t start, len, nblk, blk_base;
};

// Task record (int4): x = index of the first query in col, y = first key token,
// z = key count (1..128) | query count (1..8) << 8 | index head << 12,
// w = key-block id g * nb_cap + global block (tasks with equal w read the
// same K/V block).
struct TaskView {
  int32_t col_begin, key_start, key_len, nq, g, sub;
};
__device__ __forceinline__ TaskView decode_task(int4 t) {
  TaskView v;
  v.col_begin = t.x;
  v.key_start = t.y;
  v.key_len = t.z & 0xFF;
  v.nq = (t.z >> 8) & 0xF;
  v.g = (t.z >> 12) & 0x3;
  v.sub = t.w;
  return v;
}

// Octet-group item of the forward (int32 [kItemWords]): the tiles of one or
// two aligned octets (8 consecutive tokens of a document, positions 8k ..
// 8k+7, fewer at its end) of one query block b.
//   [0] first token of octet A, [1] first token of octet B (-1: none),
//   [2] queries of A | queries of B << 4 | index head << 8 | blocks << 12 |
//       dense << 20,
//   [3] document index,
//   [4 .. 36) uniform item (all tokens see the same blocks): the blocks
//       (document-local, ascending), then -1 to the end; dense item
//       (blocks 0 .. b, b + 1 = the block count): per token of A then of B,
//       the 64-bit mask of the blocks it selected (bit v; low word first; 0
//       past the octet's end).
constexpr int kItemWords = 36;
struct ItemView {
  int32_t tokA, tokB, nqA, nqB, g, nsel, doc;
  bool dense;
};
__device__ __forceinline__ ItemView decode_item(const int32_t* it) {
  const int4 h = *reinterpret_cast<const int4*>(it);
  ItemView v;
  v.tokA = h.x;
  v.tokB = h.y;
  v.nqA = h.z & 0xF;
  v.nqB = (h.z >> 4) & 0xF;
  v.g = (h.z >> 8) & 0x3;
  v.nsel = (h.z >> 12) & 0x7F;
  v.dense = (h.z >> 20) & 1;
  v.doc = h.w;
  return v;
}

// Index of count entry (g, doc, key block v, query block qb), v <= qb < n, in
// the order (g, doc, super-block of qb, v, qb): tasks emitted in this order
// walk one super-block of queries at a time.  Zs = super-block length in
// query blocks (>= 1).  Returns the offset inside the (g, doc) segment.
__host__ __device__ __forceinline__ int64_t tri_local(int64_t n, int64_t Zs, int64_t v,
                                                      int64_t qb) {
  const int64_t lo = (qb / Zs) * Zs;
  const int64_t hi = (lo + Zs < n) ? lo + Zs : n;
  const int64_t w = hi - lo;
  const int64_t base = lo * (lo + 1) / 2;
  int64_t offv;
  if (v < lo)
    offv = v * w;
  else
    offv = lo * w + (v - lo) * hi - (v - lo) * (v + lo - 1) / 2;
  return base + offv + (qb - (v > lo ? v : lo));
}

// Workspace layout of a plan, shared by the size query and msa_build_plan.
struct PlanLayout {
  int64_t nb_cap, tri_cap, nnz_cap, task_cap, item_cap, scan_tmp_len;
  size_t off_header, off_doc_info, off_doc_tri, off_cnt, off_off, off_col, off_tcnt, off_toff,
      off_tasks, off_scan, off_grouped, off_items, off_fflag, off_fpos, off_ftasks, off_rows,
      total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline PlanLayout plan_layout(int64_t T, int32_t D) {
  PlanLayout L{};
  // A document with n blocks holds at least 128 (n - 1) + 1 tokens, so over
  // D documents sum n <= D + (T - D) / 128, and sum n (n + 1) / 2 is largest
  // with D - 1 one-token documents and one long one.
  const int64_t x = (T - D) / kBlock + 1;
  L.nb_cap = D + (T - D) / kBlock;
  L.tri_cap = 4 * ((D - 1) + x * (x + 1) / 2);
  L.nnz_cap = int64_t(kKVHeads) * kTopK * T;
  L.task_cap = L.nnz_cap / kTaskQueries + L.tri_cap;
  // a document of n tokens has ceil(n / 8) <= n / 8 + 1 octets
  L.item_cap = int64_t(kKVHeads) * (T / 8 + D);
  // three scans' look-back status: per scan a ticket and one word per
  // 4096-element tile, 64 bits each (in 32-bit units, a multiple of 6)
  L.scan_tmp_len = 6 * (((L.tri_cap > L.task_cap ? L.tri_cap : L.task_cap) + 4095) / 4096 + 1);
  size_t o = 0;
  L.off_header = o;   o = align_up(o + sizeof(int64_t) * kHdrWords, 256);
  L.off_doc_info = o; o = align_up(o + sizeof(DocInfo) * D, 256);
  L.off_doc_tri = o;  o = align_up(o + sizeof(int64_t) * (D + 1), 256);
  L.off_cnt = o;      o = align_up(o + sizeof(int32_t) * L.tri_cap, 256);
  L.off_off = o;      o = align_up(o + sizeof(int32_t) * L.tri_cap, 256);
  L.off_col = o;      o = align_up(o + sizeof(int32_t) * L.nnz_cap, 256);
  L.off_tcnt = o;     o = align_up(o + sizeof(int32_t) * L.tri_cap, 256);
  L.off_toff = o;     o = align_up(o + sizeof(int32_t) * L.tri_cap, 256);
  L.off_tasks = o;    o = align_up(o + sizeof(int4) * L.task_cap, 256);
  L.off_scan = o;     o = align_up(o + sizeof(int32_t) * L.scan_tmp_len, 256);
  L.off_grouped = o;  o = align_up(o + sizeof(uint8_t) * kKVHeads * T, 256);
  L.off_items = o;    o = align_up(o + sizeof(int32_t) * kItemWords * L.item_cap, 256);
  L.off_fflag = o;    o = align_up(o + sizeof(int32_t) * L.task_cap, 256);
  L.off_fpos = o;     o = align_up(o + sizeof(int32_t) * L.task_cap, 256);
  L.off_ftasks = o;   o = align_up(o + sizeof(int4) * L.task_cap, 256);
  L.off_rows = o;     o = align_up(o + sizeof(int32_t) * kKVHeads * T, 256);
  L.total = o;
  return L;
}

// Programmatic dependent launch.  A kernel launched with launch_k(true, ...)
// may start while the previous kernel on the stream is still finishing (its
// launch and prologue overlap that kernel's tail); every kernel therefore
// calls grid_dep_wait() before it touches global memory, which returns once
// the previous kernel has completed and its writes are visible (at once for
// a kernel launched without the attribute; a previous kernel that never
// calls grid_dep_release() releases its dependents when it completes), and
// then grid_dep_release(), which lets the next kernel launch.  Since every
// kernel waits for its predecessor, a kernel's completion implies that of
// all before it.  Copies and event waits in the stream keep their order.
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Profiling on (msa_profile_enable): launches are then kept apart by the
// timing events and take no programmatic overlap.
bool profiling_on();
template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool overlap, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (overlap && !profiling_on()) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// A CTA's share of a persistent kernel's task list of n tasks, walked in
// chunks of C consecutive tasks (C a power of two, so the walk's index
// arithmetic stays cheap on the MMA issuer's path): full rounds of G chunks
// go round-robin over the G CTAs, so all CTAs advance through the list
// together; the tasks after the last full round are split evenly, so that
// the CTAs' counts differ by at most one task.
struct TaskWalk {
  int64_t n;      // tasks of this CTA
  int64_t full;   // of them, in full rounds
  int64_t tail0;  // first task of this CTA's share of the rest
};
template <int C>
__device__ __forceinline__ TaskWalk task_walk(int64_t ntasks) {
  const int64_t G = gridDim.x, c = blockIdx.x;
  const int64_t R = ntasks / (G * C);
  const int64_t rest = ntasks - R * G * C;
  const int64_t q = rest / G, extra = rest % G;
  TaskWalk w;
  w.full = R * C;
  w.tail0 = R * G * C + c * q + (c < extra ? c : extra);
  w.n = w.full + q + (c < extra ? 1 : 0);
  return w;
}
// Task index (into the list) of the CTA's i-th task.
template <int C>
__device__ __forceinline__ int64_t walk_task(const TaskWalk& w, int64_t i) {
  return i < w.full ? (int64_t(blockIdx.x) + (i / C) * gridDim.x) * C + (i % C)
                    : w.tail0 + (i - w.full);
}

// Kernel-launch bookkeeping (profiling hooks, launch counter) - msa_api.cu.
// launch_end counts `kernels` launches under `name`.
void launch_begin(const char* name, cudaStream_t s);
void launch_end(const char* name, cudaStream_t s, int kernels = 1);

// Launchers implemented in the kernel translation units.
cudaError_t launch_plan(const msa_plan& p, cudaStream_t s);
cudaError_t launch_forward(const msa_plan& p, const void* q, const void* k, const void* v,
                           float scale, void* o, float* lse, void* ws, cudaStream_t s);
cudaError_t launch_backward(const msa_plan& p, const void* q, const void* k, const void* v,
                            const void* o, const float* lse, const void* dout, float scale,
                            void* dq, void* dk, void* dv, void* ws, cudaStream_t s);
size_t forward_workspace_bytes(const msa_plan& p);
size_t backward_workspace_bytes(const msa_plan& p);

}  // namespace msa
