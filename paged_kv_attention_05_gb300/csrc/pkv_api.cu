// Host side of the C ABI declared in include/pkv.h: argument checks, the
// per-device workspace and error word, and the kernel launches.
#include <cuda_runtime.h>
#include <math.h>
#include <stddef.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int* err = nullptr;  // device error word
  void* ws = nullptr;  // workspace
  size_t ws_bytes = 0;
  // the step plan held in the workspace (pkv_plan / pkv_attention): its
  // geometry and the carve of the workspace it was written with
  bool plan_valid = false;
  int64_t plan_q_rows = 0, plan_bt_width = 0;
  int plan_hq = 0, plan_hkv = 0, plan_reqs = 0;
  Sizes plan_sizes{};
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
thread_local char g_msg[512] = "";

// Tracing (guarded by g_mu): event pairs around each launch while enabled.
struct TraceRec {
  int kind;
  cudaEvent_t a, b;
};
bool g_trace_on = false;
std::vector<TraceRec> g_trace;
std::vector<cudaEvent_t> g_ev_pool;
int64_t g_launches = 0;

cudaEvent_t take_event() {
  if (!g_ev_pool.empty()) {
    cudaEvent_t e = g_ev_pool.back();
    g_ev_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

template <class F>
cudaError_t traced(int kind, cudaStream_t st, F&& launch) {
  ++g_launches;
  if (!g_trace_on) return launch();
  TraceRec r{kind, take_event(), take_event()};
  cudaEventRecord(r.a, st);
  cudaError_t e = launch();
  cudaEventRecord(r.b, st);
  g_trace.push_back(r);
  return e;
}

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Device state of the current device, initialised on first use.
int current_state(DeviceState** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_NO_DEVICE, "device %d out of range", dev);
  DeviceState& s = g_dev[dev];
  if (!s.ready) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDeviceProperties");
    if (prop.major != 10 || prop.minor != 3)
      return fail(PKV_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a",
                  dev, prop.major, prop.minor);
    s.sms = prop.multiProcessorCount;
    e = cudaMalloc(&s.err, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(error word)");
    e = cudaMemset(s.err, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(error word)");
    s.ready = true;
  }
  *out = &s;
  return PKV_OK;
}

// Makes sure the workspace holds at least `z`; allocation only outside capture.
int ensure_workspace(DeviceState* s, const Sizes& z, cudaStream_t st, Workspace* ws) {
  const size_t need = workspace_bytes(z);
  if (need > s->ws_bytes) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (st != nullptr) cudaStreamIsCapturing(st, &cap);
    if (cap != cudaStreamCaptureStatusNone)
      return fail(PKV_ERR_ARG,
                  "workspace of %zu bytes needed while the stream is being captured; call "
                  "pkv_reserve_workspace before capture",
                  need);
    cudaError_t e = cudaDeviceSynchronize();  // the old workspace may still be in use
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    if (s->ws) cudaFree(s->ws);
    s->ws = nullptr;
    s->ws_bytes = 0;
    s->plan_valid = false;  // the plan lived in the old workspace
    const size_t grow = need + need / 4;
    e = cudaMalloc(&s->ws, grow);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc(workspace)");
    e = cudaMemset(s->ws, 0, grow);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(workspace)");
    s->ws_bytes = grow;
  }
  // carve for the capacity actually held, scaled from the request
  *ws = carve_workspace(s->ws, z, s->err);
  return PKV_OK;
}

int check_geometry(int32_t block_size, int32_t hkv, int32_t head_size) {
  if (hkv > 32767) return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads %d > 32767", hkv);
  if (block_size != kBlockSize)
    return fail(PKV_ERR_UNSUPPORTED, "block_size %d (only %d)", block_size, kBlockSize);
  if (head_size != kHeadSize)
    return fail(PKV_ERR_UNSUPPORTED, "head_size %d (only %d)", head_size, kHeadSize);
  if (hkv <= 0) return fail(PKV_ERR_ARG, "num_kv_heads %d", hkv);
  return PKV_OK;
}

}  // namespace

Sizes sizes_for(int64_t reqs, int64_t q_rows, int64_t bt_width, int hq, int hkv) {
  Sizes z;
  const int64_t max_keys = bt_width * kBlockSize;
  int64_t splits = (max_keys + kMinChunk - 1) / kMinChunk;
  if (splits < 1) splits = 1;
  const int group = hq / hkv;
  z.units = reqs * hkv * splits;
  z.pre = (q_rows + kPreTileQ - 1) / kPreTileQ + reqs;
  z.pairs = reqs * hkv;
  // decode query rows (tokens x heads of a group) are at most q_rows * G in
  // all and dec_rows_cap(G) per request
  const int64_t rows_a = q_rows * group, rows_b = reqs * dec_rows_cap(group);
  z.part_rows = splits * hkv * (rows_a < rows_b ? rows_a : rows_b);
  return z;
}

// Room for the plan's one-wave split of a small batch: as many decode units
// as the decode grid has workers, each with up to one unit's query rows of
// partial results (the plan takes a chunk shorter than kMinChunk only where
// the workspace holds what it makes).
Sizes with_wave_room(Sizes z, int64_t q_rows, int group, int workers) {
  if (z.units < workers) z.units = workers;
  const int64_t rows = std::min<int64_t>(dec_rows_cap(group), q_rows * group);
  if (z.part_rows < (int64_t)workers * rows) z.part_rows = (int64_t)workers * rows;
  return z;
}

size_t workspace_bytes(const Sizes& z) {
  size_t b = 256;                                      // header
  b += (size_t)z.units * sizeof(DecUnit);
  b += (size_t)z.pre * sizeof(PreEntry);
  b += (size_t)z.pairs * sizeof(SplitPair);
  b = (b + 255) & ~(size_t)255;
  b += (size_t)z.part_rows * 2 * sizeof(float);  // part_ml
  b = (b + 255) & ~(size_t)255;
  b += (size_t)z.part_rows * kHeadSize * sizeof(float);  // part_o
  return b + 256;
}

Workspace carve_workspace(void* base, const Sizes& z, int* err) {
  Workspace w;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  w.hdr = reinterpret_cast<PlanHeader*>(p);
  off += 256;
  w.units = reinterpret_cast<DecUnit*>(p + off);
  off += (size_t)z.units * sizeof(DecUnit);
  w.pre = reinterpret_cast<PreEntry*>(p + off);
  off += (size_t)z.pre * sizeof(PreEntry);
  w.pairs = reinterpret_cast<SplitPair*>(p + off);
  off += (size_t)z.pairs * sizeof(SplitPair);
  off = (off + 255) & ~(size_t)255;
  w.part_ml = reinterpret_cast<float*>(p + off);
  off += (size_t)z.part_rows * 2 * sizeof(float);
  off = (off + 255) & ~(size_t)255;
  w.part_o = reinterpret_cast<float*>(p + off);
  w.err = err;
  w.max_units = z.units;
  w.max_pre = z.pre;
  w.max_pairs = z.pairs;
  w.max_part_rows = z.part_rows;
  return w;
}

}  // namespace pkv

using namespace pkv;

extern "C" int pkv_write(const void* k, int64_t k_row_stride, const void* v,
                         int64_t v_row_stride, void* key_cache, void* value_cache,
                         int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_size, const int64_t* slot_mapping, int64_t n_tokens,
                         void* stream) {
  g_msg[0] = 0;
  int rc = check_geometry(block_size, num_kv_heads, head_size);
  if (rc) return rc;
  if (n_tokens < 0) return fail(PKV_ERR_ARG, "n_tokens %lld < 0", (long long)n_tokens);
  if (num_blocks < 1) return fail(PKV_ERR_ARG, "num_blocks %lld < 1", (long long)num_blocks);
  if (n_tokens == 0) return PKV_OK;
  if (!k || !v || !key_cache || !value_cache || !slot_mapping)
    return fail(PKV_ERR_ARG, "null pointer argument");
  const int64_t row = (int64_t)num_kv_heads * kHeadSize;
  if (k_row_stride < row || v_row_stride < row)
    return fail(PKV_ERR_ARG, "row stride below num_kv_heads * head_size (%lld)", (long long)row);
  if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache) ||
      (k_row_stride % 8) || (v_row_stride % 8))
    return fail(PKV_ERR_ALIGN, "k/v/caches must be 16-byte aligned with row strides * 2 a "
                               "multiple of 16 bytes");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  rc = current_state(&s);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = traced(0, st, [&] {
    return launch_write(static_cast<const uint16_t*>(k), k_row_stride,
                        static_cast<const uint16_t*>(v), v_row_stride,
                        static_cast<uint16_t*>(key_cache), static_cast<uint16_t*>(value_cache),
                        num_blocks, num_kv_heads, slot_mapping, n_tokens, s->err, s->sms, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "pkv_write launch");
  return PKV_OK;
}

extern "C" int pkv_write_int8(const void* k, int64_t k_row_stride, const void* v,
                              int64_t v_row_stride, void* key_cache, void* value_cache,
                              float k_scale, float v_scale, int64_t num_blocks,
                              int32_t block_size, int32_t num_kv_heads, int32_t head_size,
                              const int64_t* slot_mapping, int64_t n_tokens, void* stream) {
  g_msg[0] = 0;
  int rc = check_geometry(block_size, num_kv_heads, head_size);
  if (rc) return rc;
  if (n_tokens < 0) return fail(PKV_ERR_ARG, "n_tokens %lld < 0", (long long)n_tokens);
  if (num_blocks < 1) return fail(PKV_ERR_ARG, "num_blocks %lld < 1", (long long)num_blocks);
  if (!(k_scale > 0.f && v_scale > 0.f && k_scale < INFINITY && v_scale < INFINITY))
    return fail(PKV_ERR_ARG, "k_scale and v_scale must be finite and positive");
  if (n_tokens == 0) return PKV_OK;
  if (!k || !v || !key_cache || !value_cache || !slot_mapping)
    return fail(PKV_ERR_ARG, "null pointer argument");
  const int64_t row = (int64_t)num_kv_heads * kHeadSize;
  if (k_row_stride < row || v_row_stride < row)
    return fail(PKV_ERR_ARG, "row stride below num_kv_heads * head_size (%lld)", (long long)row);
  if (!aligned16(k) || !aligned16(v) || !aligned16(key_cache) || !aligned16(value_cache) ||
      (k_row_stride % 8) || (v_row_stride % 8))
    return fail(PKV_ERR_ALIGN, "k/v/caches must be 16-byte aligned with row strides * 2 a "
                               "multiple of 16 bytes");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  rc = current_state(&s);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = traced(0, st, [&] {
    return launch_write_int8(static_cast<const uint16_t*>(k), k_row_stride,
                             static_cast<const uint16_t*>(v), v_row_stride,
                             static_cast<int8_t*>(key_cache), static_cast<int8_t*>(value_cache),
                             num_blocks, num_kv_heads, slot_mapping, n_tokens, k_scale, v_scale,
                             s->err, s->sms, st);
  });
  if (e != cudaSuccess) return cuda_fail(e, "pkv_write_int8 launch");
  return PKV_OK;
}

namespace {

// The checks of the step metadata shared by pkv_plan and the attention calls.
int check_meta(int64_t q_rows, int32_t num_heads, int32_t num_kv_heads,
               const int32_t* query_start_loc, const int32_t* seq_lens,
               int64_t block_table_width, int32_t num_reqs) {
  if (num_kv_heads <= 0) return fail(PKV_ERR_ARG, "num_kv_heads %d", num_kv_heads);
  if (num_heads <= 0 || num_heads % num_kv_heads)
    return fail(PKV_ERR_UNSUPPORTED, "num_heads %d is not a multiple of num_kv_heads %d",
                num_heads, num_kv_heads);
  if (num_heads / num_kv_heads > kMaxGroup)
    return fail(PKV_ERR_UNSUPPORTED, "num_heads / num_kv_heads = %d > %d",
                num_heads / num_kv_heads, kMaxGroup);
  if (num_reqs < 0 || q_rows < 0 || block_table_width < 0)
    return fail(PKV_ERR_ARG, "negative size");
  if (num_reqs == 0 || q_rows == 0) return PKV_OK;
  if (!query_start_loc || !seq_lens) return fail(PKV_ERR_ARG, "null pointer argument");
  if (block_table_width < 1) return fail(PKV_ERR_ARG, "block_table_width < 1");
  if (block_table_width > kMaxBtWidth)
    return fail(PKV_ERR_UNSUPPORTED, "block_table_width %lld > %d (longest supported request is "
                "%d keys)", (long long)block_table_width, kMaxBtWidth, kMaxBtWidth * kBlockSize);
  return PKV_OK;
}

// Builds the step plan into the device workspace (state lock held).
int plan_locked(DeviceState* s, int64_t q_rows, int32_t num_heads, int32_t num_kv_heads,
                const int32_t* query_start_loc, const int32_t* seq_lens,
                int64_t block_table_width, int32_t num_reqs, int kv_int8, cudaStream_t st) {
  const int workers = decode_workers(num_heads / num_kv_heads, kv_int8, s->sms);
  const Sizes z = with_wave_room(
      sizes_for(num_reqs, q_rows, block_table_width, num_heads, num_kv_heads), q_rows,
      num_heads / num_kv_heads, workers);
  Workspace ws;
  int rc = ensure_workspace(s, z, st, &ws);
  if (rc) return rc;
  AttnArgs a{};
  a.q_rows = q_rows;
  a.hq = num_heads;
  a.hkv = num_kv_heads;
  a.qsl = query_start_loc;
  a.seq_lens = seq_lens;
  a.bt_width = block_table_width;
  a.num_reqs = num_reqs;
  a.kv_int8 = kv_int8;
  cudaError_t e = traced(1, st, [&] { return launch_plan(a, ws, workers, st); });
  if (e != cudaSuccess) return cuda_fail(e, "plan launch");
  // an int8 plan leaves prefill-class requests out: it cannot serve a bf16 call
  s->plan_valid = !kv_int8;
  s->plan_q_rows = q_rows;
  s->plan_bt_width = block_table_width;
  s->plan_hq = num_heads;
  s->plan_hkv = num_kv_heads;
  s->plan_reqs = num_reqs;
  s->plan_sizes = z;
  return PKV_OK;
}

// Runs the attention kernels of the plan held in the workspace (state lock
// held; the plan's geometry is the caller's).
int run_locked(DeviceState* s, const void* q, int64_t q_row_stride, const void* key_cache,
               const void* value_cache, int64_t num_blocks, const int32_t* block_table,
               float scale, void* out, int64_t out_row_stride, int kv_int8, float k_scale,
               float v_scale, cudaStream_t st) {
  Workspace ws = carve_workspace(s->ws, s->plan_sizes, s->err);
  AttnArgs a{};
  a.q = static_cast<const uint16_t*>(q);
  a.q_stride = q_row_stride;
  a.q_rows = s->plan_q_rows;
  a.hq = s->plan_hq;
  a.kc = static_cast<const uint16_t*>(key_cache);
  a.vc = static_cast<const uint16_t*>(value_cache);
  a.num_blocks = num_blocks;
  a.hkv = s->plan_hkv;
  a.qsl = nullptr;  // the kernels read the plan's snapshot of the metadata
  a.seq_lens = nullptr;
  a.bt = block_table;
  a.bt_width = s->plan_bt_width;
  a.num_reqs = s->plan_reqs;
  a.scale = scale;
  a.out = static_cast<uint16_t*>(out);
  a.out_stride = out_row_stride;
  a.kv_int8 = kv_int8;
  a.k_scale = kv_int8 ? k_scale : 1.f;
  a.v_scale = kv_int8 ? v_scale : 1.f;
  // Decode first.  When the step also has prefill work, the decode grid
  // leaves some SMs to it at once and the prefill grid (its programmatic
  // dependent) runs its items there beside the decode units; the prefill
  // kernel merges the split decode results at its end, once the decode grid
  // has finished (see pkv_decode.cu and pkv_prefill.cu).  An int8 call has no
  // prefill work (the plan reports such requests): its merge is a launch of
  // its own.
  cudaError_t e = traced(2, st, [&] { return launch_decode(a, ws, s->sms, st); });
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  if (kv_int8) {
    e = traced(4, st, [&] { return launch_combine(a, ws, s->sms, st); });
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  } else {
    e = traced(3, st, [&] { return launch_prefill(a, ws, s->sms, st); });
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  }
  return PKV_OK;
}

// The checks of the buffers an attention call reads and writes.
int check_buffers(const void* q, int64_t q_row_stride, int32_t num_heads, const void* key_cache,
                  const void* value_cache, int64_t num_blocks, const int32_t* block_table,
                  float scale, void* out, int64_t out_row_stride) {
  if (num_blocks < 1) return fail(PKV_ERR_ARG, "num_blocks %lld < 1", (long long)num_blocks);
  if (!q || !key_cache || !value_cache || !block_table || !out)
    return fail(PKV_ERR_ARG, "null pointer argument");
  const int64_t row = (int64_t)num_heads * kHeadSize;
  if (q_row_stride < row || out_row_stride < row)
    return fail(PKV_ERR_ARG, "q/out row stride below num_heads * head_size (%lld)",
                (long long)row);
  if (!aligned16(q) || !aligned16(out) || !aligned16(key_cache) || !aligned16(value_cache) ||
      (q_row_stride % 8) || (out_row_stride % 8))
    return fail(PKV_ERR_ALIGN, "q/out/caches must be 16-byte aligned with row strides * 2 a "
                               "multiple of 16 bytes");
  if (!(scale == scale)) return fail(PKV_ERR_ARG, "scale is NaN");
  return PKV_OK;
}

// pkv_attention and pkv_attention_int8: kv_int8 = 0 for bf16 caches, 1 for
// int8 codes with the two scales (decode-class requests only).
int attention_common(const void* q, int64_t q_row_stride, int64_t q_rows, int32_t num_heads,
                     const void* key_cache, const void* value_cache, int64_t num_blocks,
                     int32_t block_size, int32_t num_kv_heads, int32_t head_size,
                     const int32_t* query_start_loc, const int32_t* seq_lens,
                     const int32_t* block_table, int64_t block_table_width, int32_t num_reqs,
                     float scale, void* out, int64_t out_row_stride, void* stream, int kv_int8,
                     float k_scale, float v_scale) {
  g_msg[0] = 0;
  int rc = check_geometry(block_size, num_kv_heads, head_size);
  if (rc) return rc;
  rc = check_meta(q_rows, num_heads, num_kv_heads, query_start_loc, seq_lens,
                  block_table_width, num_reqs);
  if (rc) return rc;
  if (num_blocks < 1) return fail(PKV_ERR_ARG, "num_blocks %lld < 1", (long long)num_blocks);
  if (num_reqs == 0 || q_rows == 0) return PKV_OK;
  rc = check_buffers(q, q_row_stride, num_heads, key_cache, value_cache, num_blocks, block_table,
                     scale, out, out_row_stride);
  if (rc) return rc;
  if (kv_int8 && !(k_scale > 0.f && v_scale > 0.f && k_scale < INFINITY && v_scale < INFINITY))
    return fail(PKV_ERR_ARG, "k_scale and v_scale must be finite and positive");

  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  rc = current_state(&s);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  rc = plan_locked(s, q_rows, num_heads, num_kv_heads, query_start_loc, seq_lens,
                   block_table_width, num_reqs, kv_int8, st);
  if (rc) return rc;
  return run_locked(s, q, q_row_stride, key_cache, value_cache, num_blocks, block_table, scale,
                    out, out_row_stride, kv_int8, k_scale, v_scale, st);
}

}  // namespace

extern "C" int pkv_plan(int64_t q_rows, int32_t num_heads, int32_t num_kv_heads,
                        const int32_t* query_start_loc, const int32_t* seq_lens,
                        int64_t block_table_width, int32_t num_reqs, void* stream) {
  g_msg[0] = 0;
  int rc = check_meta(q_rows, num_heads, num_kv_heads, query_start_loc, seq_lens,
                      block_table_width, num_reqs);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  rc = current_state(&s);
  if (rc) return rc;
  if (num_reqs == 0 || q_rows == 0) {  // an empty step: nothing to plan, nothing to run
    s->plan_valid = true;
    s->plan_q_rows = q_rows;
    s->plan_reqs = 0;
    s->plan_hq = num_heads;
    s->plan_hkv = num_kv_heads;
    s->plan_bt_width = block_table_width;
    return PKV_OK;
  }
  return plan_locked(s, q_rows, num_heads, num_kv_heads, query_start_loc, seq_lens,
                     block_table_width, num_reqs, 0, static_cast<cudaStream_t>(stream));
}

extern "C" int pkv_attention_planned(const void* q, int64_t q_row_stride, int32_t num_heads,
                                     const void* key_cache, const void* value_cache,
                                     int64_t num_blocks, int32_t block_size,
                                     int32_t num_kv_heads, int32_t head_size,
                                     const int32_t* block_table, float scale, void* out,
                                     int64_t out_row_stride, void* stream) {
  g_msg[0] = 0;
  int rc = check_geometry(block_size, num_kv_heads, head_size);
  if (rc) return rc;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  rc = current_state(&s);
  if (rc) return rc;
  if (!s->plan_valid)
    return fail(PKV_ERR_ARG, "no step plan on this device (call pkv_plan or pkv_attention first)");
  if (num_heads != s->plan_hq || num_kv_heads != s->plan_hkv)
    return fail(PKV_ERR_ARG, "num_heads %d / num_kv_heads %d differ from the plan's %d / %d",
                num_heads, num_kv_heads, s->plan_hq, s->plan_hkv);
  if (s->plan_reqs == 0 || s->plan_q_rows == 0) return PKV_OK;
  rc = check_buffers(q, q_row_stride, num_heads, key_cache, value_cache, num_blocks, block_table,
                     scale, out, out_row_stride);
  if (rc) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the decode and prefill kernels take work from two cursors in the plan
  // header, which the plan kernel zeroes; a further run of the same plan
  // zeroes them again first (a stream-ordered memset, graph-capturable)
  PlanHeader* hdr = carve_workspace(s->ws, s->plan_sizes, s->err).hdr;
  static_assert(offsetof(PlanHeader, pre_counter) == offsetof(PlanHeader, dec_counter) + 4,
                "adjacent cursors");
  cudaError_t e = cudaMemsetAsync(&hdr->dec_counter, 0, 2 * sizeof(int), st);
  if (e != cudaSuccess) return cuda_fail(e, "cursor reset");
  return run_locked(s, q, q_row_stride, key_cache, value_cache, num_blocks, block_table, scale,
                    out, out_row_stride, 0, 1.f, 1.f, st);
}

extern "C" int pkv_attention(const void* q, int64_t q_row_stride, int64_t q_rows,
                             int32_t num_heads, const void* key_cache, const void* value_cache,
                             int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                             int32_t head_size, const int32_t* query_start_loc,
                             const int32_t* seq_lens, const int32_t* block_table,
                             int64_t block_table_width, int32_t num_reqs, float scale, void* out,
                             int64_t out_row_stride, void* stream) {
  return attention_common(q, q_row_stride, q_rows, num_heads, key_cache, value_cache, num_blocks,
                          block_size, num_kv_heads, head_size, query_start_loc, seq_lens,
                          block_table, block_table_width, num_reqs, scale, out, out_row_stride,
                          stream, 0, 1.f, 1.f);
}

extern "C" int pkv_attention_int8(const void* q, int64_t q_row_stride, int64_t q_rows,
                                  int32_t num_heads, const void* key_cache,
                                  const void* value_cache, float k_scale, float v_scale,
                                  int64_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                  int32_t head_size, const int32_t* query_start_loc,
                                  const int32_t* seq_lens, const int32_t* block_table,
                                  int64_t block_table_width, int32_t num_reqs, float scale,
                                  void* out, int64_t out_row_stride, void* stream) {
  return attention_common(q, q_row_stride, q_rows, num_heads, key_cache, value_cache, num_blocks,
                          block_size, num_kv_heads, head_size, query_start_loc, seq_lens,
                          block_table, block_table_width, num_reqs, scale, out, out_row_stride,
                          stream, 1, k_scale, v_scale);
}

extern "C" int pkv_reserve_workspace(int32_t max_reqs, int64_t max_q_rows,
                                     int64_t block_table_width, int32_t num_heads,
                                     int32_t num_kv_heads) {
  g_msg[0] = 0;
  if (max_reqs < 0 || max_q_rows < 0 || block_table_width < 0 || num_kv_heads <= 0 ||
      num_heads <= 0 || num_heads % num_kv_heads)
    return fail(PKV_ERR_ARG, "bad sizes");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc) return rc;
  Workspace ws;
  const int group = num_heads / num_kv_heads;
  const int workers = std::max(decode_workers(group, 0, s->sms), decode_workers(group, 1, s->sms));
  return ensure_workspace(s, with_wave_room(sizes_for(max_reqs, max_q_rows, block_table_width,
                                                      num_heads, num_kv_heads),
                                            max_q_rows, group, workers),
                          nullptr, &ws);
}

extern "C" int pkv_workspace_size(int32_t max_reqs, int64_t max_q_rows,
                                  int64_t block_table_width, int32_t num_heads,
                                  int32_t num_kv_heads, int32_t num_sms,
                                  pkv_workspace_info* info) {
  g_msg[0] = 0;
  if (!info) return fail(PKV_ERR_ARG, "info is null");
  if (max_reqs < 0 || max_q_rows < 0 || block_table_width < 0 || num_kv_heads <= 0 ||
      num_heads <= 0 || num_heads % num_kv_heads || num_sms <= 0)
    return fail(PKV_ERR_ARG, "bad sizes");
  const int group = num_heads / num_kv_heads;
  const int w16 = decode_workers(group, 0, num_sms), w8 = decode_workers(group, 1, num_sms);
  // what pkv_reserve_workspace holds: room for both cache types' plans
  const Sizes z = with_wave_room(
      sizes_for(max_reqs, max_q_rows, block_table_width, num_heads, num_kv_heads), max_q_rows,
      group, std::max(w16, w8));
  info->bytes = (int64_t)workspace_bytes(z);
  info->decode_units = z.units;
  info->prefill_tiles = z.pre;
  info->split_pairs = z.pairs;
  info->partial_rows = z.part_rows;
  info->decode_workers = w16;
  info->decode_workers_int8 = w8;
  return PKV_OK;
}

extern "C" int pkv_get_error(void* stream, int32_t* bits) {
  g_msg[0] = 0;
  if (!bits) return fail(PKV_ERR_ARG, "bits is null");
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PKV_ERR_NO_DEVICE, "device %d out of range", dev);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  // the word of the allocating calls (only if one ran on this device: a
  // device no allocating call has used gets no state, and nothing is
  // allocated here), then the word of pkv_attention_noalloc
  int v = 0;
  DeviceState& s = g_dev[dev];
  if (s.ready) {
    e = cudaMemcpy(&v, s.err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read error word");
    e = cudaMemset(s.err, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear error word");
  }
  int w = 0;
  const int ce = noalloc_take_error(dev, &w);
  if (ce) return cuda_fail(static_cast<cudaError_t>(ce), "read the no-alloc error word");
  *bits = v | w;
  return PKV_OK;
}

extern "C" const char* pkv_last_error_string(void) { return g_msg; }

extern "C" int pkv_num_sms(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  if (current_state(&s)) return -1;
  return s->sms;
}

extern "C" int pkv_prepare_step(const int32_t* query_start_loc, const int32_t* num_computed,
                                const int32_t* idx_mapping, const int32_t* persistent_block_table,
                                int64_t persistent_rows, int64_t block_table_width,
                                int32_t num_reqs, int64_t num_tokens_padded, int64_t* positions,
                                int32_t* seq_lens, int64_t* slot_mapping, int32_t* block_table,
                                void* stream) {
  g_msg[0] = 0;
  if (num_reqs < 0 || num_tokens_padded < 0 || block_table_width < 1 || persistent_rows < 0)
    return fail(PKV_ERR_ARG, "negative size or empty block-table row");
  if (num_reqs == 0 && num_tokens_padded == 0) return PKV_OK;
  if (!positions || !slot_mapping || (num_reqs > 0 && (!query_start_loc || !num_computed ||
                                                       !persistent_block_table || !seq_lens)))
    return fail(PKV_ERR_ARG, "null pointer argument");
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState* s = nullptr;
  int rc = current_state(&s);
  if (rc) return rc;
  PrepArgs p;
  p.qsl = query_start_loc;
  p.num_computed = num_computed;
  p.idx = idx_mapping;
  p.pbt = persistent_block_table;
  p.pbt_rows = persistent_rows;
  p.bt_width = block_table_width;
  p.num_reqs = num_reqs;
  p.num_tokens_padded = num_tokens_padded;
  p.positions = positions;
  p.seq_lens = seq_lens;
  p.slot_mapping = slot_mapping;
  p.block_table = block_table;
  p.err = s->err;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = traced(5, st, [&] { return launch_prepare(p, s->sms, st); });
  if (e != cudaSuccess) return cuda_fail(e, "prepare launch");
  return PKV_OK;
}

extern "C" int pkv_trace_enable(int on) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_trace_on = on != 0;
  return PKV_OK;
}

extern "C" int pkv_trace_read(double* ms, int64_t* launches, int n) {
  std::lock_guard<std::mutex> lock(g_mu);
  double tot[PKV_TRACE_KINDS] = {};  // NOLINT
  int64_t cnt[PKV_TRACE_KINDS] = {};
  int rc = PKV_OK;
  for (const TraceRec& r : g_trace) {
    float t = 0.f;
    cudaError_t e = cudaEventSynchronize(r.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, r.a, r.b);
    if (e != cudaSuccess) rc = cuda_fail(e, "trace event");
    if (r.kind >= 0 && r.kind < PKV_TRACE_KINDS) {
      tot[r.kind] += t;
      cnt[r.kind] += 1;
    }
    g_ev_pool.push_back(r.a);
    g_ev_pool.push_back(r.b);
  }
  g_trace.clear();
  for (int i = 0; i < n && i < PKV_TRACE_KINDS; ++i) {
    if (ms) ms[i] = tot[i];
    if (launches) launches[i] = cnt[i];
  }
  return rc == PKV_OK ? PKV_TRACE_KINDS : rc;
}

extern "C" int64_t pkv_launch_count(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  return g_launches;
}
