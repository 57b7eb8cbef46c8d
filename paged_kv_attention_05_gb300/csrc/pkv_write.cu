// Cache-write scatter: the step's new K/V rows into the block-paged cache.
//
// "vLLM 推理全流程深度解析" (vLLM inference deep dive), reshape_and_cache
// section: a negative slot is skipped; otherwise block = slot / block_size,
// offset = slot % block_size and the token's [num_kv_heads, head_size] rows
// land at cache[block][offset].  "Tour: One forward pass", stop 4: padding
// rows carry PAD_SLOT_ID = -1.
//
// GB300 layout of the work: the copy is pure HBM traffic (read 2 rows, write
// 2 rows per token), so a warp moves one 2 KB piece of a token's contiguous
// [num_kv_heads * 128] K row and the same piece of its V row: the slot is
// read once, the lanes take consecutive 16-byte vectors, four of each row per
// lane, all loads issued before the stores (fully coalesced 512-byte
// transactions, and enough bytes in flight per SM to cover HBM latency).  The
// grid is a multiple of the SM count and strides over (token, piece).
//
// Both write kernels are launched with programmatic stream serialisation:
// their CTAs may be scheduled while the kernel before them (typically the
// previous step's attention, which reads the cache) finishes, and wait for
// it in grid_dep_wait() before touching any memory; then they let the next
// kernel (the step plan, which waits for this one in turn) start its set-up.
#include "pkv_internal.cuh"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256) write_kernel(const uint16_t* __restrict__ k,
                                                    int64_t k_stride,
                                                    const uint16_t* __restrict__ v,
                                                    int64_t v_stride, uint16_t* __restrict__ kc,
                                                    uint16_t* __restrict__ vc, int64_t num_slots,
                                                    int row_vecs, const int64_t* __restrict__ slots,
                                                    int64_t n_tokens, int* err) {
  grid_dep_wait();
  grid_dep_launch();
  // row_vecs = 16-byte vectors per token row = num_kv_heads * 128 * 2 / 16
  constexpr int kUnroll = 4;
  constexpr int kPiece = 32 * kUnroll;  // vectors of a row one warp moves
  const int pieces = (row_vecs + kPiece - 1) / kPiece;
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t units = n_tokens * pieces;
  for (int64_t w = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; w < units;
       w += nwarps) {
    const int64_t t = w / pieces;
    const int base = (int)(w - t * pieces) * kPiece;
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (lane == 0 && base == 0) atomicOr(err, PKV_DEV_ERR_SLOT_RANGE);
      continue;
    }
    // cache row of this slot: [block][offset] == slot * row (contiguous pool)
    const uint4* ks = reinterpret_cast<const uint4*>(k + t * k_stride);
    const uint4* vs = reinterpret_cast<const uint4*>(v + t * v_stride);
    uint4* kd = reinterpret_cast<uint4*>(kc + slot * (int64_t)row_vecs * 8);
    uint4* vd = reinterpret_cast<uint4*>(vc + slot * (int64_t)row_vecs * 8);
    {
      uint4 kv[kUnroll], vv[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int e = base + u * 32 + lane;
        if (e < row_vecs) {
          kv[u] = __ldg(ks + e);
          vv[u] = __ldg(vs + e);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int e = base + u * 32 + lane;
        if (e < row_vecs) {
          kd[e] = kv[u];
          vd[e] = vv[u];
        }
      }
    }
  }
}

// The same scatter into int8 caches: each thread turns 16 bf16 values (two
// 16-byte loads) into 16 codes (one 16-byte store), code = clamp(rne(x /
// scale), -127, 127) in fp32 with the IEEE division (a NaN value gives 0).
__device__ __forceinline__ uint32_t quant4(uint32_t lo, uint32_t hi, float scale) {
  const float x[4] = {__uint_as_float(lo << 16), __uint_as_float(lo & 0xFFFF0000u),
                      __uint_as_float(hi << 16), __uint_as_float(hi & 0xFFFF0000u)};
  uint32_t w = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float r = rintf(__fdiv_rn(x[i], scale));
    r = (r == r) ? fminf(fmaxf(r, -127.f), 127.f) : 0.f;
    w |= ((uint32_t)(int)r & 0xFFu) << (8 * i);
  }
  return w;
}

__global__ void __launch_bounds__(256) write_int8_kernel(
    const uint16_t* __restrict__ k, int64_t k_stride, const uint16_t* __restrict__ v,
    int64_t v_stride, int8_t* __restrict__ kc, int8_t* __restrict__ vc, int64_t num_slots,
    int row_vecs, const int64_t* __restrict__ slots, int64_t n_tokens, float k_scale,
    float v_scale, int* err) {
  grid_dep_wait();
  grid_dep_launch();
  // row_vecs = 16-code vectors per token row = num_kv_heads * 128 / 16
  const int64_t per_token = 2 * (int64_t)row_vecs;
  const int64_t total = n_tokens * per_token;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / per_token;
    const int rem = (int)(i - t * per_token);
    const bool is_v = rem >= row_vecs;
    const int vec = is_v ? rem - row_vecs : rem;
    const int64_t slot = __ldg(slots + t);
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (rem == 0) atomicOr(err, PKV_DEV_ERR_SLOT_RANGE);
      continue;
    }
    const uint16_t* src = (is_v ? v + t * v_stride : k + t * k_stride) + (int64_t)vec * 16;
    int8_t* dst = (is_v ? vc : kc) + slot * (int64_t)row_vecs * 16 + (int64_t)vec * 16;
    const float sc = is_v ? v_scale : k_scale;
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
    *reinterpret_cast<uint4*>(dst) =
        make_uint4(quant4(a.x, a.y, sc), quant4(a.z, a.w, sc), quant4(b.x, b.y, sc),
                   quant4(b.z, b.w, sc));
  }
}

}  // namespace

cudaError_t launch_write_int8(const uint16_t* k, int64_t k_stride, const uint16_t* v,
                              int64_t v_stride, int8_t* kc, int8_t* vc, int64_t num_blocks,
                              int hkv, const int64_t* slots, int64_t n_tokens, float k_scale,
                              float v_scale, int* err, int sms, cudaStream_t st) {
  const int row_vecs = hkv * kHeadSize / 16;
  const int64_t total = n_tokens * 2 * (int64_t)row_vecs;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = (int64_t)sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_dependent(write_int8_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, k,
                          k_stride, v, v_stride, kc, vc, num_blocks * kBlockSize, row_vecs, slots,
                          n_tokens, k_scale, v_scale, err);
}

cudaError_t launch_write(const uint16_t* k, int64_t k_stride, const uint16_t* v, int64_t v_stride,
                         uint16_t* kc, uint16_t* vc, int64_t num_blocks, int hkv,
                         const int64_t* slots, int64_t n_tokens, int* err, int sms,
                         cudaStream_t st) {
  const int row_vecs = hkv * kHeadSize * 2 / 16;
  const int threads = 256;
  const int64_t units = n_tokens * ((row_vecs + 127) / 128);  // a warp per 128-vector piece
  int64_t blocks = (units + threads / 32 - 1) / (threads / 32);
  const int64_t cap = (int64_t)sms * 8;  // 8 resident 256-thread CTAs per SM
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return launch_dependent(write_kernel, dim3((unsigned)blocks), dim3(threads), 0, st, k, k_stride,
                          v, v_stride, kc, vc, num_blocks * kBlockSize, row_vecs, slots, n_tokens,
                          err);
}

}  // namespace pkv
