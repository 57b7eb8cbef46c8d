// Prefill / chunked-prefill attention (requests with more than one query
// token) on the 5th-generation tensor cores: tcgen05.mma with accumulators in
// tensor memory, K/V pages gathered by TMA through the block table.
//
// What it computes: "Tour: One forward pass", stop 10 — causal attention for
// the request's query rows over all of its keys (R3: 298 query rows, 298
// keys), the keys found through the block table; stop 3 — query row i sits
// at position num_computed + i, so a chunk that continues a cached prompt sees
// the cached keys plus its own causal triangle.  "vLLM 推理全流程深度解析",
// prefill section: lower-triangular causal mask; the FlashAttention idea of
// keeping the score tile on chip.  "vLLM MHA Code Path: From QKV to Paged KV
// Cache", "One Path Covers MHA, GQA, and MQA": query head h reads KV head
// h / (Hq / Hkv).
//
// GB300 design.  One work item = (request, 128-row query tile, query head);
// a persistent grid (one CTA per SM, 512 TMEM columns each) takes items from
// an atomic cursor in the order the plan wrote them.  Inside a CTA:
//   warp 0      TMA producer: the Q tile once per item; per 128-key tile,
//               the 8 K pages and 8 V pages (each page a 16-slot x 64-dim
//               box, two per page for the two 64-dim halves, 128-byte
//               swizzle) into a 2-stage ring; in the last tile of a request
//               it zero-fills V rows past seq_len so that no stale value
//               (NaN) reaches the P.V product;
//   warp 1      allocates TMEM and issues the MMAs from one thread:
//               S = Q K^T (M = N = 128, K = 128 in 8 steps of 16) into one of
//               two TMEM score buffers, then O += P V (P from shared memory,
//               V read MN-major) into the TMEM output buffer; tcgen05.commit
//               signals the mbarriers;
//   warps 4-7   softmax, one query row per thread (TMEM lane = row): load
//               the 128 scores of the row, causal/length mask, running max in
//               the log2 domain, exp2, row sum, P as bf16 into shared memory
//               (the operand layout of the next MMA).  The output in TMEM is
//               rescaled only when a row's max grows by more than 2^8, which
//               is exact (softmax is shift invariant) and rare; the final
//               division by the row sum happens in the epilogue, which writes
//               the bf16 rows of the item straight to global memory.
// Every mbarrier wait is bounded; on expiry the kernel records
// PKV_DEV_ERR_TIMEOUT, stops issuing work, frees its TMEM and returns.
#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int kThreads = 256;
constexpr int kStages = 2;
constexpr int kTileK = 128;                       // keys per KV tile
constexpr int kHalfBytes = 128 * 128;             // 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kHalfBytes;        // Q, K, V or P tile: 32 KB
constexpr int kPageBoxBytes = 16 * 128;           // one 16-slot x 64-dim box
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;         // log2 units

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffP = kOffV + kStages * kTileBytes;
constexpr int kOffBar = kOffP + kTileBytes;
// barriers: q_full, k_full[2], v_full[2], v_tma[2], kv_empty[2], s_full[2],
// p_full, o_done  (15 x 8 bytes), then the TMEM address and control words
constexpr int kNumBars = 15;
constexpr int kOffCtl = kOffBar + kNumBars * 8;
constexpr int kSmemBytes = kOffCtl + 64 + 1024;  // + alignment slack

enum { B_Q = 0, B_K = 1, B_V = 3, B_VT = 5, B_EMPTY = 7, B_S = 9, B_P = 11, B_O = 12 };

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// Shared-memory matrix descriptor: 128-byte swizzle, SBO = 1024 bytes
// (8-row groups), LBO as given (MN-major: distance between 64-element atoms).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((1024 >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M = N = 128.
__host__ __device__ constexpr uint32_t idesc_bf16(bool b_mn_major) {
  return (1u << 4)                       // D format f32
         | (1u << 7)                     // A format bf16
         | (1u << 10)                    // B format bf16
         | ((b_mn_major ? 1u : 0u) << 16)  // B major-ness
         | ((128u >> 3) << 17)           // N
         | ((128u >> 4) << 24);          // M
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
      : "memory");
}

#define PKV_LD32(taddr, v)                                                                     \
  asm volatile(                                                                                \
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"   \
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),   \
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),            \
        "=f"(v[13]), "=f"(v[14]), "=f"(v[15]), "=f"(v[16]), "=f"(v[17]), "=f"(v[18]),         \
        "=f"(v[19]), "=f"(v[20]), "=f"(v[21]), "=f"(v[22]), "=f"(v[23]), "=f"(v[24]),         \
        "=f"(v[25]), "=f"(v[26]), "=f"(v[27]), "=f"(v[28]), "=f"(v[29]), "=f"(v[30]),         \
        "=f"(v[31])                                                                            \
      : "r"(taddr))

#define PKV_ST32(taddr, v)                                                                     \
  asm volatile(                                                                                \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12," \
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"  \
      ::"r"(taddr), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),        \
      "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]), "f"(v[12]),         \
      "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]), "f"(v[18]), "f"(v[19]),     \
      "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]), "f"(v[24]), "f"(v[25]), "f"(v[26]),     \
      "f"(v[27]), "f"(v[28]), "f"(v[29]), "f"(v[30]), "f"(v[31])                              \
      : "memory")

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

struct Item {
  int r, qt, h, g;
  int q0, n, L, ctx;
  int nkv;
};

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, AttnArgs a, Workspace ws) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  volatile int* ctl = reinterpret_cast<volatile int*>(smem + kOffCtl);
  // ctl[0] = TMEM base address, ctl[1] = abort flag, ctl[2] = current item
  volatile int* abort = ctl + 1;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.hq / a.hkv;

  if (tid == 0) {
    mbar_init(bar(B_Q), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(B_K + s), 1);
      mbar_init(bar(B_V + s), 1);
      mbar_init(bar(B_VT + s), 1);
      mbar_init(bar(B_EMPTY + s), 1);
      mbar_init(bar(B_S + s), 1);
    }
    mbar_init(bar(B_P), 128);
    mbar_init(bar(B_O), 1);
    ctl[1] = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                     sbase + kOffCtl),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)ctl[0];
  const uint32_t tm_s0 = tmem, tm_o = tmem + 256;

  const int n_items = ws.hdr->n_pre_entries * a.hq;
  uint32_t tile_base = 0;  // KV tiles processed by this CTA so far (all items)
  uint32_t item_cnt = 0;
  uint32_t vt_uses[kStages] = {0, 0};

  for (;;) {
    if (tid == 0) ctl[2] = atomicAdd(&ws.hdr->pre_counter, 1);
    __syncthreads();
    const int w = ctl[2];
    if (w >= n_items || *abort) break;
    Item it;
    {
      const PreEntry e = ws.pre[w / a.hq];
      it.r = e.r;
      it.qt = e.qt;
      it.h = w % a.hq;
      it.g = it.h / G;
      it.nkv = e.nkv;
      it.q0 = a.qsl[it.r];
      it.n = a.qsl[it.r + 1] - it.q0;
      it.L = a.seq_lens[it.r];
      it.ctx = it.L - it.n;
    }
    const int* btrow = a.bt + (int64_t)it.r * a.bt_width;

    if (warp == 0) {
      // ---------------- TMA producer ----------------
      if (lane == 0) {
        mbar_expect_tx(bar(B_Q), kTileBytes);
        const int row0 = it.q0 + it.qt * kPreTileQ;
        tma_load_3d(sbase + kOffQ, &tm_q, bar(B_Q), 0, it.h, row0);
        tma_load_3d(sbase + kOffQ + kHalfBytes, &tm_q, bar(B_Q), 64, it.h, row0);
      }
      for (int j = 0; j < it.nkv; ++j) {
        const uint32_t c = tile_base + j;
        const int s = c % kStages;
        if (c >= (uint32_t)kStages) {
          if (!mbar_wait_warp(bar(B_EMPTY + s), ((c / kStages) - 1) & 1, abort, ws.err)) break;
        }
        const int key0 = j * kTileK;
        const int pages = min(8, (it.L - key0 + 15) / 16);
        const bool tail = key0 + kTileK > it.L;
        const uint32_t kdst = sbase + kOffK + s * kTileBytes;
        const uint32_t vdst = sbase + kOffV + s * kTileBytes;
        if (lane == 0) {
          mbar_expect_tx(bar(B_K + s), pages * 2 * kPageBoxBytes);
          for (int p = 0; p < pages; ++p) {
            int blk = __ldg(btrow + (key0 >> 4) + p);
            if (blk < 0 || (int64_t)blk >= a.num_blocks) {
              atomicOr(ws.err, PKV_DEV_ERR_BLOCK_ID);
              blk = 0;
            }
            tma_load_4d(kdst + p * kPageBoxBytes, &tm_k, bar(B_K + s), 0, it.g, 0, blk);
            tma_load_4d(kdst + kHalfBytes + p * kPageBoxBytes, &tm_k, bar(B_K + s), 64, it.g, 0,
                        blk);
          }
          const uint32_t vbar = tail ? bar(B_VT + s) : bar(B_V + s);
          mbar_expect_tx(vbar, pages * 2 * kPageBoxBytes);
          for (int p = 0; p < pages; ++p) {
            int blk = __ldg(btrow + (key0 >> 4) + p);
            if (blk < 0 || (int64_t)blk >= a.num_blocks) blk = 0;
            tma_load_4d(vdst + p * kPageBoxBytes, &tm_v, vbar, 0, it.g, 0, blk);
            tma_load_4d(vdst + kHalfBytes + p * kPageBoxBytes, &tm_v, vbar, 64, it.g, 0, blk);
          }
        }
        if (tail) {
          // wait for the V boxes, zero the rows of keys >= seq_len, publish
          const bool ok = mbar_wait_warp(bar(B_VT + s), vt_uses[s] & 1, abort, ws.err);
          vt_uses[s]++;
          if (!ok) break;
          const int z0 = it.L - key0;  // first key row to clear
          const int chunks = (kTileK - z0) * 16;
          uint8_t* v = smem + kOffV + s * kTileBytes;
          for (int i = lane; i < chunks; i += 32) {
            const int row = z0 + (i >> 4), within = i & 15;
            const int half = within >> 3, ch = within & 7;
            *reinterpret_cast<uint4*>(v + half * kHalfBytes + row * 128 + ch * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_V + s));
        }
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer ----------------
      if (lane == 0) {
        const uint32_t id_s = idesc_bf16(false), id_o = idesc_bf16(true);
        const uint32_t qa = sbase + kOffQ;
        auto issue_s = [&](uint32_t c) -> bool {
          const int s = c % kStages;
          if (!mbar_wait(bar(B_K + s), (c / kStages) & 1, abort, ws.err)) return false;
          tc_fence_after();
          const uint32_t kb = sbase + kOffK + s * kTileBytes;
          const uint32_t d = tm_s0 + (c & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            mma_bf16(d, sdesc(qa + off, 16), sdesc(kb + off, 16), id_s, kk > 0);
          }
          mma_commit(bar(B_S + (c & 1)));
          return true;
        };
        bool ok = mbar_wait(bar(B_Q), item_cnt & 1, abort, ws.err);
        if (ok) ok = issue_s(tile_base);
        for (int j = 0; ok && j < it.nkv; ++j) {
          const uint32_t c = tile_base + j;
          const int s = c % kStages;
          if (j + 1 < it.nkv && !issue_s(c + 1)) break;
          if (!mbar_wait(bar(B_P), c & 1, abort, ws.err)) break;
          if (!mbar_wait(bar(B_V + s), (c / kStages) & 1, abort, ws.err)) break;
          tc_fence_after();
          const uint32_t pa = sbase + kOffP, vb = sbase + kOffV + s * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t aoff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            const uint32_t boff = kk * 16 * 128;  // 16 key rows per step
            mma_bf16(tm_o, sdesc(pa + aoff, 16), sdesc(vb + boff, kHalfBytes), id_o,
                     (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(bar(B_O));
          mma_commit(bar(B_EMPTY + s));
        }
      }
      __syncwarp();
    } else if (warp >= 4) {
      // ---------------- softmax + epilogue, one row per thread ----------------
      const int row = tid - 128;  // == 32 * (warp % 4) + lane == TMEM lane
      const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
      const int qrow = it.qt * kPreTileQ + row;  // row inside the request
      const bool valid_row = qrow < it.n;
      const int qpos = valid_row ? it.ctx + qrow : 0;  // last visible key
      const float sl2 = a.scale * kLog2e;
      float m_used = -INFINITY, l_sum = 0.f;
      uint8_t* P = smem + kOffP;
      bool ok = true;
      for (int j = 0; j < it.nkv; ++j) {
        const uint32_t c = tile_base + j;
        if (!mbar_wait_warp(bar(B_S + (c & 1)), (c >> 1) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[128];
        const uint32_t sa = tm_s0 + (c & 1) * 128 + lane_off;
        PKV_LD32(sa + 0, (sv + 0));
        PKV_LD32(sa + 32, (sv + 32));
        PKV_LD32(sa + 64, (sv + 64));
        PKV_LD32(sa + 96, (sv + 96));
        tmem_wait_ld();
        const int key0 = j * kTileK;
        const int lim = qpos - key0;  // columns <= lim are visible
        float mt = -INFINITY;
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          sv[i] = (i <= lim) ? sv[i] * sl2 : -INFINITY;
          mt = fmaxf(mt, sv[i]);
        }
        float alpha = 1.f;
        bool resc = false;
        if (mt > m_used + kRescaleThreshold) {
          alpha = fast_exp2(m_used - mt);  // 0 on the first tile
          resc = (j > 0);
          m_used = mt;
        }
        float rs = 0.f;
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          sv[i] = fast_exp2(sv[i] - m_used);
          rs += sv[i];
        }
        l_sum = l_sum * alpha + rs;
        if (j > 0) {
          // the previous P.V must be complete before P and O are touched
          if (!mbar_wait_warp(bar(B_O), (c - 1) & 1, abort, ws.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (__any_sync(0xffffffffu, resc)) {
            float ov[32];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              const uint32_t oa = tm_o + ch * 32 + lane_off;
              PKV_LD32(oa, ov);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] *= alpha;
              PKV_ST32(oa, ov);
            }
            tmem_wait_st();
          }
        }
        // P row (bf16) in the 128-byte swizzled K-major layout
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          uint4 pk;
          pk.x = pack_bf16(sv[ch * 8 + 0], sv[ch * 8 + 1]);
          pk.y = pack_bf16(sv[ch * 8 + 2], sv[ch * 8 + 3]);
          pk.z = pack_bf16(sv[ch * 8 + 4], sv[ch * 8 + 5]);
          pk.w = pack_bf16(sv[ch * 8 + 6], sv[ch * 8 + 7]);
          const int half = ch >> 3, c8 = ch & 7;
          *reinterpret_cast<uint4*>(P + half * kHalfBytes + row * 128 +
                                    ((c8 ^ (row & 7)) << 4)) = pk;
        }
        fence_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_P));
      }
      if (ok) {
        const uint32_t c_last = tile_base + it.nkv - 1;
        if (mbar_wait_warp(bar(B_O), c_last & 1, abort, ws.err)) {
          tc_fence_after();
          const float inv = 1.f / l_sum;
          uint16_t* orow = a.out + (int64_t)(it.q0 + qrow) * a.out_stride +
                           (int64_t)it.h * kHeadSize;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            float ov[32];
            PKV_LD32(tm_o + ch * 32 + lane_off, ov);
            tmem_wait_ld();
            if (valid_row) {
#pragma unroll
              for (int i = 0; i < 32; i += 8) {
                uint4 pk;
                pk.x = pack_bf16(ov[i + 0] * inv, ov[i + 1] * inv);
                pk.y = pack_bf16(ov[i + 2] * inv, ov[i + 3] * inv);
                pk.z = pack_bf16(ov[i + 4] * inv, ov[i + 5] * inv);
                pk.w = pack_bf16(ov[i + 6] * inv, ov[i + 7] * inv);
                *reinterpret_cast<uint4*>(orow + ch * 32 + i) = pk;
              }
            }
          }
        }
      }
    }
    tile_base += it.nkv;
    item_cnt++;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(kTmemCols));
  }
}

}  // namespace

cudaError_t launch_prefill(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  CUtensorMap tq, tk, tv;
  if (!make_rows_map(&tq, a.q, a.q_rows, a.hq, a.q_stride, 1, kPreTileQ) ||
      !make_cache_map(&tk, a.kc, a.num_blocks, a.hkv) ||
      !make_cache_map(&tv, a.vc, a.num_blocks, a.hkv))
    return cudaErrorInvalidValue;
  prefill_kernel<<<sms, kThreads, kSmemBytes, st>>>(tq, tk, tv, a, ws);
  return cudaGetLastError();
}

}  // namespace pkv
