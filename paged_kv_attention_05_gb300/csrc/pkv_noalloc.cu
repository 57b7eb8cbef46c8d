// pkv_attention_noalloc: the attention call for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc: services that fix their device-memory
// footprint when they start and must not grow it afterwards, hosts whose
// device memory is handed out by an allocator of their own that the library
// must not bypass, and latency-critical loops that cannot afford the device
// synchronisation a cudaMalloc/cudaFree pair implies.  pkv_attention grows a
// workspace with cudaMalloc on first use; this entry point runs the same
// kernels on the same step plan with their scratch (step plan, work lists,
// split-KV partial results) in one file-scope device array of fixed size
// instead, and allocates nothing.
//
// The array is a static __device__ object: every GPU that loads the library
// holds kScratchBytes of it until the process exits.  In host code its name
// is only a host-side stand-in, so the device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call on that device.  Every call shares the array and it keeps the
// previous call's contents; the plan kernel rewrites the work lists and
// resets the scheduler cursors at the start of each call, which is all that
// must start from zero.  Calls whose kernels overlap on the GPU (for example
// on two streams) race on the array.  The device error word of these calls
// lives beside the array; pkv_get_error reads and clears it together with the
// allocating calls' word.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr size_t kScratchBytes = 32u << 20;  // 32 MiB

__device__ __align__(256) uint8_t g_scratch[kScratchBytes];
__device__ __align__(256) int g_scratch_err;  // device error word of this entry point

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_scratch_ptr[kMaxDevices];
int* g_err_ptr[kMaxDevices];
int g_sms[kMaxDevices];

// The refusal reasons below are for readers of this file; the caller gets
// the code only (pkv_last_error_string belongs to the allocating calls).
int noalloc_fail(int code, const char* reason) {
  (void)reason;
  return code;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" int pkv_attention_noalloc(const void* q, int64_t q_row_stride, int64_t q_rows,
                                     int32_t num_heads, const void* key_cache,
                                     const void* value_cache, int64_t num_blocks,
                                     int32_t block_size, int32_t num_kv_heads,
                                     int32_t head_size, const int32_t* query_start_loc,
                                     const int32_t* seq_lens, const int32_t* block_table,
                                     int64_t block_table_width, int32_t num_reqs, float scale,
                                     void* out, int64_t out_row_stride, void* stream) {
  // same argument contract as pkv_attention
  if (block_size != kBlockSize || head_size != kHeadSize)
    return noalloc_fail(PKV_ERR_UNSUPPORTED, "block_size must be 16 and head_size 128");
  // a decode unit packs the KV head into 16 bits (with the query-token count)
  if (num_kv_heads > 32767) return noalloc_fail(PKV_ERR_UNSUPPORTED, "num_kv_heads > 32767");
  if (num_kv_heads <= 0 || num_heads <= 0 || num_heads % num_kv_heads)
    return noalloc_fail(PKV_ERR_UNSUPPORTED, "num_heads must be a multiple of num_kv_heads");
  if (num_heads / num_kv_heads > kMaxGroup)
    return noalloc_fail(PKV_ERR_UNSUPPORTED, "num_heads / num_kv_heads above 32");
  if (num_reqs < 0 || q_rows < 0 || block_table_width < 0 || num_blocks < 1)
    return noalloc_fail(PKV_ERR_ARG, "negative size or empty pool");
  if (num_reqs == 0 || q_rows == 0) return PKV_OK;
  if (!q || !key_cache || !value_cache || !query_start_loc || !seq_lens || !block_table || !out)
    return noalloc_fail(PKV_ERR_ARG, "null pointer argument");
  if (block_table_width < 1 || block_table_width > kMaxBtWidth)
    return noalloc_fail(PKV_ERR_UNSUPPORTED, "block_table_width outside [1, 32768]");
  const int64_t row = (int64_t)num_heads * kHeadSize;
  if (q_row_stride < row || out_row_stride < row)
    return noalloc_fail(PKV_ERR_ARG, "q/out row stride below num_heads * head_size");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(out) |
       reinterpret_cast<uintptr_t>(key_cache) | reinterpret_cast<uintptr_t>(value_cache)) & 15 ||
      (q_row_stride % 8) || (out_row_stride % 8))
    return noalloc_fail(PKV_ERR_ALIGN, "q/out/caches must be 16-byte aligned, strides too");
  if (!(scale == scale)) return noalloc_fail(PKV_ERR_ARG, "scale is NaN");

  // the scratch this call can need, by the same bound pkv_attention sizes
  // its workspace with; above the static array's size the call is refused
  const int group = num_heads / num_kv_heads;
  const Sizes z = sizes_for(num_reqs, q_rows, block_table_width, num_heads, num_kv_heads);
  const size_t need = workspace_bytes(z);
  if (need > kScratchBytes)
    return noalloc_fail(PKV_ERR_UNSUPPORTED, "batch needs more scratch than the static array");

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return noalloc_fail(PKV_ERR_NO_DEVICE, "no current CUDA device");
  void* scratch = nullptr;
  int* err = nullptr;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_scratch_ptr[dev]) {
      // once per device, with the device current: the array's device address
      int major = 0, minor = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          major != 10 || minor != 3)
        return noalloc_fail(PKV_ERR_NO_DEVICE, "current device is not sm_103");
      int n = 0;
      if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return noalloc_fail(PKV_ERR_CUDA, "cudaDeviceGetAttribute failed");
      void* p = nullptr;
      void* pe = nullptr;
      e = cudaGetSymbolAddress(&p, g_scratch);
      if (e != cudaSuccess) return noalloc_fail(PKV_ERR_CUDA, "cudaGetSymbolAddress(scratch)");
      e = cudaGetSymbolAddress(&pe, g_scratch_err);
      if (e != cudaSuccess) return noalloc_fail(PKV_ERR_CUDA, "cudaGetSymbolAddress(error)");
      g_sms[dev] = n;
      g_err_ptr[dev] = static_cast<int*>(pe);
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
    err = g_err_ptr[dev];
    sms = g_sms[dev];
  }

  // The plan of pkv_attention: a workspace for z plus room for a small
  // batch's one-wave split (shorter split chunks, more units and partial
  // rows), carved the same way, so that both calls make the same plan and the
  // same bits.  Where that room does not fit beside z, the plan holds no more
  // than z: a small batch may then take fewer, longer splits than
  // pkv_attention, with the same result up to fp32 rounding.
  Sizes zc = with_wave_room(z, q_rows, group, decode_workers(group, 0, sms));
  if (workspace_bytes(zc) > kScratchBytes) zc = z;
  Workspace ws = carve_workspace(scratch, zc, err);
  AttnArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.q_stride = q_row_stride;
  a.q_rows = q_rows;
  a.hq = num_heads;
  a.kc = static_cast<const uint16_t*>(key_cache);
  a.vc = static_cast<const uint16_t*>(value_cache);
  a.num_blocks = num_blocks;
  a.hkv = num_kv_heads;
  a.qsl = query_start_loc;
  a.seq_lens = seq_lens;
  a.bt = block_table;
  a.bt_width = block_table_width;
  a.num_reqs = num_reqs;
  a.scale = scale;
  a.out = static_cast<uint16_t*>(out);
  a.out_stride = out_row_stride;
  a.kv_int8 = 0;
  a.k_scale = a.v_scale = 1.f;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the kernels of pkv_attention, one after the other on the caller's stream
  if ((e = launch_plan(a, ws, decode_workers(group, 0, sms), st)) != cudaSuccess ||
      (e = launch_decode(a, ws, sms, st)) != cudaSuccess ||
      (e = launch_prefill(a, ws, sms, st)) != cudaSuccess)  // (merges the splits at its end)
    return noalloc_fail(PKV_ERR_CUDA, "kernel launch failed");
  return PKV_OK;
}

namespace pkv {

int noalloc_take_error(int dev, int* bits) {
  *bits = 0;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (dev < 0 || dev >= kMaxDevices || !g_err_ptr[dev]) return 0;  // never used on dev
  int v = 0;
  cudaError_t e = cudaMemcpy(&v, g_err_ptr[dev], sizeof(int), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(g_err_ptr[dev], 0, sizeof(int));
  if (e != cudaSuccess) return (int)e;
  *bits = v;
  return 0;
}

}  // namespace pkv
