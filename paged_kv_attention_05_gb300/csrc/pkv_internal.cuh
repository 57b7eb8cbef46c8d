// Internal declarations shared by the CUDA translation units of libpkv.
// Not part of the public C ABI (include/pkv.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "pkv.h"

namespace pkv {

constexpr int kHeadSize = 128;   // elements per head row
constexpr int kBlockSize = 16;   // tokens per cache block (page)
constexpr int kMaxGroup = 32;    // query heads per KV head handled by one decode unit
constexpr int kDecTile = 64;     // split-KV chunks are whole multiples of this many keys
constexpr int kMinChunk = 256;   // smallest split-KV chunk (tokens)
constexpr int kMaxChunk = 2048;  // largest split-KV chunk (tokens)
constexpr int kMaxBtWidth = 32768;  // block-table entries per request (524,288 keys) at most
constexpr int kPreTileQ = 128;   // query rows per prefill tile

// Query rows a decode unit can carry (query tokens x heads of one KV head).
__host__ __device__ constexpr int dec_rows_cap(int group) { return group <= 16 ? 16 : 32; }

// The work lists are a snapshot of the request metadata taken by the plan
// kernel: the attention kernels read query_start_loc and seq_lens only
// through them, so a plan can serve several layers (and later changes of the
// metadata arrays cannot send a kernel out of bounds).

// One decode work unit (32 bytes): request r with qn query tokens starting at
// row q0 (ctx keys before the first one), KV head g, keys [k0, k1) of the
// request; gq = g | qn << 16.  Split results occupy partial rows part .. part
// + qn * G - 1 (row = token * G + head in group).
struct __align__(16) DecUnit {
  int r, gq, ctx, nsplit, k0, k1, part, q0;
};

// One prefill work entry: request r (n query rows from q0, seq_len L),
// 128-row query tile qt; nkv = number of 128-key tiles it reads (the work
// estimate used for longest-first ordering).
struct __align__(16) PreEntry {
  int r, qt, nkv, q0;
  int n, L, pad0, pad1;
};

// A (request, KV head) whose keys were split over several decode units: split
// s keeps its qn * G partial rows from first + s * qn * G; the request's
// rows start at q0.
struct __align__(16) SplitPair {
  int r, g, first, nsplit;
  int q0, qn, pad0, pad1;
};

// Header of the step plan, written by the plan kernel each call.
struct PlanHeader {
  int n_dec_units;
  int n_pre_entries;
  int dec_counter;  // dynamic scheduler cursors, reset by the plan kernel
  int pre_counter;
  int chunk;
  int n_pairs;      // split pairs to merge
  int max_rows;     // most query rows of one split pair (qn * G)
  int pre_tiles;    // 128-key tiles of all prefill entries (one query head pair each)
  int pre_max_tiles;  // key tiles of the longest prefill entry
  int pad[7];
};

// Device pointers into the per-device workspace.
struct Workspace {
  PlanHeader* hdr;
  DecUnit* units;
  PreEntry* pre;
  SplitPair* pairs;  // [max_reqs * hkv] split pairs (n_pairs used)
  float* part_ml;    // [part rows][2]: running max (log2 domain) and sum
  float* part_o;     // [part rows][128]: unnormalised output
  int* err;          // device error word
  int64_t max_units;
  int64_t max_pre;
  int64_t max_pairs;
  int64_t max_part_rows;
};

// Bytes needed for a workspace serving up to these sizes.
// Capacities of a workspace for a call (or a reservation) of these sizes.
struct Sizes {
  int64_t units, pre, pairs, part_rows;
};
Sizes sizes_for(int64_t reqs, int64_t q_rows, int64_t bt_width, int hq, int hkv);
size_t workspace_bytes(const Sizes& z);
// z grown to hold a small batch's one-wave split: one decode unit per worker,
// each with up to one unit's query rows of partial results.
Sizes with_wave_room(Sizes z, int64_t q_rows, int group, int workers);
// Reads and clears the device error word of pkv_attention_noalloc on device
// dev (0 when that call never ran there); returns 0 or a cudaError_t.
// Allocates nothing.
int noalloc_take_error(int dev, int* bits);
Workspace carve_workspace(void* base, const Sizes& z, int* err);

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current
// device, once per device (each device holds its own copy of the kernel and
// of the attribute); `done` is the kernel's own flag array.
constexpr int kMaxAttrDevices = 64;
template <typename Kernel>
cudaError_t smem_attr_once(Kernel* kernel, int bytes, std::atomic<bool>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxAttrDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

// Launchers (return cudaGetLastError()).
cudaError_t launch_write(const uint16_t* k, int64_t k_stride, const uint16_t* v, int64_t v_stride,
                         uint16_t* kc, uint16_t* vc, int64_t num_blocks, int hkv,
                         const int64_t* slots, int64_t n_tokens, int* err, int sms,
                         cudaStream_t st);
cudaError_t launch_write_int8(const uint16_t* k, int64_t k_stride, const uint16_t* v,
                              int64_t v_stride, int8_t* kc, int8_t* vc, int64_t num_blocks,
                              int hkv, const int64_t* slots, int64_t n_tokens, float k_scale,
                              float v_scale, int* err, int sms, cudaStream_t st);

struct AttnArgs {
  const uint16_t* q;
  int64_t q_stride;
  int64_t q_rows;
  int hq;
  const uint16_t* kc;
  const uint16_t* vc;
  int64_t num_blocks;
  int hkv;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* bt;
  int64_t bt_width;
  int num_reqs;
  float scale;
  uint16_t* out;
  int64_t out_stride;
  // int8 caches (kc / vc then point at int8 codes): K = code * k_scale,
  // V = code * v_scale; decode-class requests only
  int kv_int8;
  float k_scale;
  float v_scale;
};

// TMA descriptors (pkv_tma.cu).  rows map: [rows, heads, 128] bf16 with a row
// stride, box = 64 columns x box_heads x box_rows; cache map: [num_blocks, 16,
// hkv, 128] bf16, box = 64 columns x 1 head x 16 slots x 1 block.  Both use
// the 128-byte swizzle.
bool tma_available();
// int8 cache map: [num_blocks, 16, hkv, 128] int8, box = 128 codes x 1 head x
// 16 slots x 1 block (one 2 KB box per page), 128-byte swizzle.
bool make_cache_map_i8(CUtensorMap* m, const void* base, int64_t num_blocks, int hkv);
bool make_rows_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int64_t row_stride,
                   int box_heads, int box_rows);
bool make_cache_map(CUtensorMap* m, const void* base, int64_t num_blocks, int hkv);

struct PrepArgs {
  const int32_t* qsl;           // [num_reqs + 1]
  const int32_t* num_computed;  // [num_reqs]
  const int32_t* idx;           // [num_reqs] persistent row of each batch row, or null
  const int32_t* pbt;           // [pbt_rows, bt_width] persistent block-table rows
  int64_t pbt_rows;
  int64_t bt_width;
  int num_reqs;
  int64_t num_tokens_padded;
  int64_t* positions;           // [num_tokens_padded]
  int32_t* seq_lens;            // [num_reqs]
  int64_t* slot_mapping;        // [num_tokens_padded]
  int32_t* block_table;         // [num_reqs, bt_width], or null
  int* err;
};
cudaError_t launch_prepare(const PrepArgs& p, int sms, cudaStream_t st);

cudaError_t launch_plan(const AttnArgs& a, const Workspace& ws, int dec_grid, cudaStream_t st);
cudaError_t launch_decode(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st);
// the decode path over int8 caches (pkv_decode_i8.cu)
cudaError_t launch_decode_i8(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st);
cudaError_t launch_combine(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st);
// Independent decode workers (warps) the decode grid runs for a head grouping
// and cache type; the plan sizes its split chunks for this many.
int decode_workers(int group, int kv_int8, int sms);
int decode_i8_warps(int group);
cudaError_t launch_prefill(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st);

// Programmatic dependent launch.  The cache write and the attention kernels
// (plan, decode, prefill; the merge for int8 calls) are launched with programmatic stream
// serialisation: a kernel's CTAs may start while the kernel before it in the
// stream is still running, do their set-up (barriers, shared-memory
// clearing), and then wait in grid_dep_wait() until that kernel has finished
// and its writes are visible, before reading anything it produced.  Each such
// kernel waits before it finishes, so finishing implies that every kernel
// before it has finished too.  (The prefill kernel, the decode kernel's
// dependent, reads the plan without waiting, since the decode grid triggers
// it after its own wait for the plan, and waits for the decode grid only
// before its final merge: its items run beside the decode units.)
// Launched without the attribute, the wait returns at once.
template <typename... Params, typename... Args>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

#ifdef __CUDACC__
// Waits until the kernel before this one in the stream has finished and its
// memory is visible (a no-op without programmatic serialisation).
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}
// Lets the next kernel in the stream start its set-up; it still waits for
// this kernel to finish before it reads what this kernel writes.
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}
#endif

}  // namespace pkv
