// Split-KV decode attention over the paged cache (requests with one query
// token), with the split merge fused into the last unit of each
// (request, KV head) to finish.
//
// What it computes: "vLLM 推理全流程深度解析" (vLLM inference deep dive),
// paged_attention_v1 section — find the request's physical blocks through
// block_tables, load K/V block by block into shared memory, dot-product the
// query with each key, online softmax, weighted sum of V.  "Tour: One forward
// pass", stop 10: R1 reads 541 keys — the step's own token, written by the
// cache update first, included.  "vLLM MHA Code Path: From QKV to Paged KV
// Cache", section "One Path Covers MHA, GQA, and MQA": the G = Hq / Hkv query
// heads of a KV head read the same K/V rows.
//
// GB300 design.  Decode is bound by HBM: every key and value row is read once
// per KV head and used by the G query heads of that KV head.
//   * Work unit = (request, KV head, key range of at most 1024 keys); the plan
//     kernel lists the units.  One CTA per SM runs until the list is empty.
//   * Warp 4 is the producer.  It takes units from an atomic cursor, fetches
//     the unit's block ids with the whole warp, and streams the unit's pages
//     with TMA (one 16-slot x 64-dim box per page, K and V, two 64-dim halves,
//     128-byte swizzle) into a ring of 64-key stages (4 pages).  It does not
//     wait for the consumers at unit boundaries, so the ring stays full across
//     units; the unit's G query rows come with the unit descriptor, also by
//     TMA, into one of two query slots.
//   * Warps 0-3 consume: warp w takes page w of every stage.  The G query
//     heads are the rows of 16-row tiles, so S = Q.K^T and O += P.V run on the
//     tensor cores with bf16 mma.sync m16n8k16 and fp32 accumulation (with up
//     to 32 heads per K/V row the FMA pipes could not keep pace with HBM);
//     the running max and sum stay in registers, with quad shuffles for the
//     row reductions and exp2 with the scale folded in.  Keys at or past the
//     unit's end are masked in S and their V values zeroed in the fragments,
//     so stale or NaN cache slots never reach the product.
//   * At the end of a unit the four warps merge through shared memory.  A
//     unit that is one split of several writes (max, sum, unnormalised output)
//     in fp32 to the workspace and takes a ticket; the split that arrives last
//     merges all splits (the weights staged in shared memory, then one output
//     column per thread with independent loads) and writes the bf16 result.
//     No CTA ever waits on another; every mbarrier wait is bounded.
#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int kConsumers = 4;                    // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;  // + one producer warp
constexpr int kHalf = kDecTile * 128;            // 64 keys x 64 dims (8 KB)
constexpr int kStageBytes = 4 * kHalf;           // K lo | K hi | V lo | V hi
constexpr int kPageHalf = kBlockSize * 128;      // one TMA box: 16 slots x 64 dims
constexpr int kMaxUnitPages = kMaxChunk / kBlockSize;

template <int MT>
struct Cfg {
  static constexpr int kStages = MT == 1 ? 5 : 4;
  static constexpr int kRows = MT * 16;                  // query rows per tile
  static constexpr int kQHalf = kRows * 128;             // one 64-dim half of a query slot
  static constexpr int kQSlot = 2 * kQHalf;
  static constexpr int kMerge = kConsumers * kRows * (kHeadSize + 2) * 4;
  // layout (from a 1024-byte aligned base)
  static constexpr int kOffStage = 0;
  static constexpr int kOffQ = kOffStage + kStages * kStageBytes;
  static constexpr int kOffMerge = kOffQ + 2 * kQSlot;
  static constexpr int kOffUnit = kOffMerge + kMerge;     // 2 x (DecUnit + block ids)
  static constexpr int kUnitSlot = 32 + kMaxUnitPages * 4;
  static constexpr int kOffBar = (kOffUnit + 2 * kUnitSlot + 7) & ~7;
  static constexpr int kNumBars = 2 * kStages + 4;         // full, empty, ufull[2], uempty[2]
  static constexpr int kOffCtl = kOffBar + kNumBars * 8;
  static constexpr int kSmem = kOffCtl + 32 + 1024;
};

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col); bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;\n" ::"n"(kConsumers * 32) : "memory");
}

// keep the bf16 halves of a register whose token index is below `valid`
__device__ __forceinline__ uint32_t mask_pair(uint32_t v, int tok_lo, int valid) {
  const uint32_t lo = tok_lo < valid ? 0x0000FFFFu : 0u;
  const uint32_t hi = tok_lo + 1 < valid ? 0xFFFF0000u : 0u;
  return v & (lo | hi);
}

template <int MT>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, AttnArgs a, Workspace ws) {
  using C = Cfg<MT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kOffBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (C::kStages + s); };
  auto ufull_bar = [&](int s) { return bar0 + 8u * (2 * C::kStages + s); };
  auto uempty_bar = [&](int s) { return bar0 + 8u * (2 * C::kStages + 2 + s); };
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kOffCtl);
  int* s_ticket = reinterpret_cast<int*>(smem + C::kOffCtl + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.hq / a.hkv;
  const int n_units = ws.hdr->n_dec_units;

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), kConsumers);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(ufull_bar(s), 1);
      mbar_init(uempty_bar(s), kConsumers);
    }
    *abort = 0;
    fence_barrier_init();
  }
  // query rows G..kRows-1 of both slots are never loaded: keep them zero
  for (int i = tid; i < 2 * 2 * C::kRows * 8; i += kThreads) {
    const int c = i & 7, row = (i >> 3) % C::kRows, half = (i >> 3) / C::kRows;  // half 0..3
    if (row >= G)
      *reinterpret_cast<uint4*>(smem + C::kOffQ + half * C::kQHalf + row * 128 + c * 16) =
          make_uint4(0, 0, 0, 0);
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ------------------------------ producer ------------------------------
    uint32_t tile_cnt = 0, unit_cnt = 0;
    for (;; ++unit_cnt) {
      int u = 0;
      if (lane == 0) u = atomicAdd(&ws.hdr->dec_counter, 1);
      u = __shfl_sync(0xffffffffu, u, 0);
      const int slot = unit_cnt & 1;
      if (unit_cnt >= 2 &&
          !mbar_wait_warp(uempty_bar(slot), ((unit_cnt >> 1) - 1) & 1, abort, ws.err))
        break;
      uint8_t* us = smem + C::kOffUnit + slot * C::kUnitSlot;
      DecUnit* ud = reinterpret_cast<DecUnit*>(us);
      int* ids = reinterpret_cast<int*>(us + 32);
      if (u >= n_units) {
        if (lane == 0) {
          ud->r = -1;
          mbar_arrive(ufull_bar(slot));
        }
        break;
      }
      const DecUnit un = ws.units[u];
      const int* btrow = a.bt + (int64_t)un.r * a.bt_width;
      const int p0 = un.k0 / kBlockSize;
      const int npages = (un.k1 + kBlockSize - 1) / kBlockSize - p0;
      for (int i = lane; i < npages; i += 32) {
        int blk = __ldg(btrow + p0 + i);
        if (blk < 0 || (int64_t)blk >= a.num_blocks) {
          atomicOr(ws.err, PKV_DEV_ERR_BLOCK_ID);
          blk = 0;
        }
        ids[i] = blk;
      }
      if (lane == 0) *ud = un;
      __syncwarp();
      if (lane == 0) {
        // the unit's query rows: heads g*G .. g*G+G-1 of token query_start_loc[r]
        const int q0 = a.qsl[un.r];
        const uint32_t qdst = sbase + C::kOffQ + slot * C::kQSlot;
        mbar_expect_tx(ufull_bar(slot), 2 * G * 128);
        tma_load_3d(qdst, &tm_q, ufull_bar(slot), 0, un.g * G, q0);
        tma_load_3d(qdst + C::kQHalf, &tm_q, ufull_bar(slot), 64, un.g * G, q0);
      }
      const int ntiles = (un.k1 - un.k0 + kDecTile - 1) / kDecTile;
      bool ok = true;
      for (int t = 0; t < ntiles; ++t, ++tile_cnt) {
        const int s = tile_cnt % C::kStages;
        if (tile_cnt >= (uint32_t)C::kStages &&
            !mbar_wait_warp(empty_bar(s), ((tile_cnt / C::kStages) - 1) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const int pages = min(4, npages - t * 4);
          const uint32_t st = sbase + C::kOffStage + s * kStageBytes;
          mbar_expect_tx(full_bar(s), pages * 4 * kPageHalf);
          for (int p = 0; p < pages; ++p) {
            const int blk = ids[t * 4 + p];
            const uint32_t off = p * kPageHalf;
            tma_load_4d(st + off, &tm_k, full_bar(s), 0, un.g, 0, blk);
            tma_load_4d(st + kHalf + off, &tm_k, full_bar(s), 64, un.g, 0, blk);
            tma_load_4d(st + 2 * kHalf + off, &tm_v, full_bar(s), 0, un.g, 0, blk);
            tma_load_4d(st + 3 * kHalf + off, &tm_v, full_bar(s), 64, un.g, 0, blk);
          }
        }
        __syncwarp();
      }
      if (!ok) break;
    }
    return;
  }

  // ------------------------------ consumers ------------------------------
  const int gid = lane >> 2, tig = lane & 3;
  const int mi = lane >> 3, rr = lane & 7;
  const float sl2 = a.scale * kLog2e;
  float* mw = reinterpret_cast<float*>(smem + C::kOffMerge);
  float* lw = mw + kConsumers * C::kRows;
  float* ow = lw + kConsumers * C::kRows;
  uint32_t tile_cnt = 0;
  for (uint32_t unit_cnt = 0;; ++unit_cnt) {
    const int slot = unit_cnt & 1;
    if (!mbar_wait_warp(ufull_bar(slot), (unit_cnt >> 1) & 1, abort, ws.err)) break;
    const DecUnit un = *reinterpret_cast<const DecUnit*>(smem + C::kOffUnit + slot * C::kUnitSlot);
    if (un.r < 0) break;
    const uint32_t qs = sbase + C::kOffQ + slot * C::kQSlot;
    const int k0 = un.k0, k1 = un.k1;
    const int ntiles = (k1 - k0 + kDecTile - 1) / kDecTile;

    float o[MT][16][4];
    float m_run[MT][2], l_run[MT][2];
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
      for (int dn = 0; dn < 16; ++dn)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][dn][e] = 0.f;
      m_run[mt][0] = m_run[mt][1] = -INFINITY;
      l_run[mt][0] = l_run[mt][1] = 0.f;
    }

    bool ok = true;
    for (int t = 0; t < ntiles; ++t, ++tile_cnt) {
      const int s = tile_cnt % C::kStages;
      if (!mbar_wait_warp(full_bar(s), (tile_cnt / C::kStages) & 1, abort, ws.err)) {
        ok = false;
        break;
      }
      const int pos0 = k0 + t * kDecTile + warp * 16;
      if (pos0 < k1) {
        const int valid = k1 - pos0;  // keys of this page inside the unit (may be >= 16)
        const uint32_t st = sbase + C::kOffStage + s * kStageBytes;
        const int prow = warp * 16;   // first row of this warp's page in the stage
        // S = Q K^T for the page's 16 keys (two n-tiles of 8)
        float sacc[MT][2][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.f;
#pragma unroll
        for (int kstep = 0; kstep < 8; ++kstep) {
          const int half = kstep >> 2, c0 = (kstep & 3) * 2;
          uint32_t b0, b1, b2, b3;
          {
            const int krow = prow + rr + ((mi >> 1) << 3);
            ldsm_x4(st + half * kHalf + sw128(krow, c0 + (mi & 1)), b0, b1, b2, b3);
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            uint32_t a0, a1, a2, a3;
            const int qrow = mt * 16 + rr + ((mi & 1) << 3);
            ldsm_x4(qs + half * C::kQHalf + sw128(qrow, c0 + (mi >> 1)), a0, a1, a2, a3);
            mma_bf16(sacc[mt][0], a0, a1, a2, a3, b0, b1);
            mma_bf16(sacc[mt][1], a0, a1, a2, a3, b2, b3);
          }
        }

        // online softmax (log2 domain), masking keys >= k1
        uint32_t pa[MT][4];
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          float x[2][4];
          float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tok = nt * 8 + tig * 2 + (e & 1);
              x[nt][e] = tok < valid ? sacc[mt][nt][e] * sl2 : -INFINITY;
            }
            mx0 = fmaxf(mx0, fmaxf(x[nt][0], x[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(x[nt][2], x[nt][3]));
          }
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
          const float mn0 = fmaxf(m_run[mt][0], mx0), mn1 = fmaxf(m_run[mt][1], mx1);
          const float al0 = fast_exp2(m_run[mt][0] - mn0), al1 = fast_exp2(m_run[mt][1] - mn1);
          m_run[mt][0] = mn0;
          m_run[mt][1] = mn1;
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            x[nt][0] = fast_exp2(x[nt][0] - mn0);
            x[nt][1] = fast_exp2(x[nt][1] - mn0);
            x[nt][2] = fast_exp2(x[nt][2] - mn1);
            x[nt][3] = fast_exp2(x[nt][3] - mn1);
            s0 += x[nt][0] + x[nt][1];
            s1 += x[nt][2] + x[nt][3];
          }
          l_run[mt][0] = l_run[mt][0] * al0 + s0;
          l_run[mt][1] = l_run[mt][1] * al1 + s1;
#pragma unroll
          for (int dn = 0; dn < 16; ++dn) {
            o[mt][dn][0] *= al0;
            o[mt][dn][1] *= al0;
            o[mt][dn][2] *= al1;
            o[mt][dn][3] *= al1;
          }
          pa[mt][0] = pack_bf16(x[0][0], x[0][1]);
          pa[mt][1] = pack_bf16(x[0][2], x[0][3]);
          pa[mt][2] = pack_bf16(x[1][0], x[1][1]);
          pa[mt][3] = pack_bf16(x[1][2], x[1][3]);
        }

        // O += P V (V rows read transposed); zero V of keys past the unit
#pragma unroll
        for (int dn = 0; dn < 16; dn += 2) {
          const int half = dn >> 3, c = dn & 7;
          uint32_t b0, b1, b2, b3;
          const int vrow = prow + rr + ((mi & 1) << 3);
          ldsm_x4_t(st + (2 + half) * kHalf + sw128(vrow, c + (mi >> 1)), b0, b1, b2, b3);
          if (valid < 16) {
            b0 = mask_pair(b0, 2 * tig, valid);
            b2 = mask_pair(b2, 2 * tig, valid);
            b1 = mask_pair(b1, 8 + 2 * tig, valid);
            b3 = mask_pair(b3, 8 + 2 * tig, valid);
          }
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            mma_bf16(o[mt][dn], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b0, b1);
            mma_bf16(o[mt][dn + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(s));
    }
    if (!ok) break;
    __syncwarp();
    if (lane == 0) mbar_arrive(uempty_bar(slot));  // query slot free for the producer

    // merge the four warps' states: [warp][row] m, l and [warp][row][128] o
    constexpr int ROWS = C::kRows;
    consumer_sync();  // the merge buffer is free (previous unit done with it)
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      float l0 = l_run[mt][0], l1 = l_run[mt][1];
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      const int ra = mt * 16 + gid, rb = ra + 8;
      if (tig == 0) {
        mw[warp * ROWS + ra] = m_run[mt][0];
        mw[warp * ROWS + rb] = m_run[mt][1];
        lw[warp * ROWS + ra] = l0;
        lw[warp * ROWS + rb] = l1;
      }
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {
        const int col = dn * 8 + tig * 2;
        *reinterpret_cast<float2*>(ow + (warp * ROWS + ra) * kHeadSize + col) =
            make_float2(o[mt][dn][0], o[mt][dn][1]);
        *reinterpret_cast<float2*>(ow + (warp * ROWS + rb) * kHeadSize + col) =
            make_float2(o[mt][dn][2], o[mt][dn][3]);
      }
    }
    consumer_sync();

    const int d = tid;  // one output column per consumer thread
    const int q0 = a.qsl[un.r];
    uint16_t* out_row = a.out + (int64_t)q0 * a.out_stride + (int64_t)un.g * G * kHeadSize + d;
    if (un.nsplit == 1) {
      for (int row = 0; row < G; ++row) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, mw[w * ROWS + row]);
        float acc = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) {
          const float f = fast_exp2(mw[w * ROWS + row] - M);
          acc += f * ow[(w * ROWS + row) * kHeadSize + d];
          lsum += f * lw[w * ROWS + row];
        }
        out_row[row * kHeadSize] = __bfloat16_as_ushort(__float2bfloat16_rn(acc / lsum));
      }
      continue;
    }
    for (int row = 0; row < G; ++row) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, mw[w * ROWS + row]);
      float acc = 0.f, lsum = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float f = fast_exp2(mw[w * ROWS + row] - M);
        acc += f * ow[(w * ROWS + row) * kHeadSize + d];
        lsum += f * lw[w * ROWS + row];
      }
      const int64_t prow = (int64_t)un.part * G + row;
      ws.part_o[prow * kHeadSize + d] = acc;
      if (d == 0) {
        ws.part_ml[prow * 2] = M;
        ws.part_ml[prow * 2 + 1] = lsum;
      }
    }
    __threadfence();
    consumer_sync();
    if (tid == 0) *s_ticket = atomicAdd(&ws.counters[(int64_t)un.r * a.hkv + un.g], 1);
    consumer_sync();
    if (*s_ticket != un.nsplit - 1) continue;

    // the last split to finish merges all splits of (r, g)
    __threadfence();
    const int first = un.part - un.split, ns = un.nsplit;
    float* wm = mw;              // [ns][G] weights
    float* wl = mw + ns * G;     // [G] 1 / total sum
    consumer_sync();             // everyone is past the reads of mw/lw/ow above
    for (int i = tid; i < ns * G; i += kConsumers * 32)
      wm[i] = __ldcg(ws.part_ml + ((int64_t)first * G + i) * 2);
    consumer_sync();
    if (tid < G) {
      float M = -INFINITY;
      for (int s = 0; s < ns; ++s) M = fmaxf(M, wm[s * G + tid]);
      float lsum = 0.f;
      for (int s = 0; s < ns; ++s) {
        const float f = fast_exp2(wm[s * G + tid] - M);
        lsum += f * __ldcg(ws.part_ml + ((int64_t)(first + s) * G + tid) * 2 + 1);
        wm[s * G + tid] = f;
      }
      wl[tid] = 1.f / lsum;
    }
    consumer_sync();
    for (int row = 0; row < G; ++row) {
      float acc = 0.f;
      const float* po = ws.part_o + ((int64_t)first * G + row) * kHeadSize + d;
#pragma unroll 8
      for (int s = 0; s < ns; ++s) acc += wm[s * G + row] * __ldcg(po + (int64_t)s * G * kHeadSize);
      out_row[row * kHeadSize] = __bfloat16_as_ushort(__float2bfloat16_rn(acc * wl[row]));
    }
  }
}

template <int MT>
cudaError_t launch_mt(const AttnArgs& a, const Workspace& ws, int grid, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<MT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg<MT>::kSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const int G = a.hq / a.hkv;
  CUtensorMap tq, tk, tv;
  if (!make_rows_map(&tq, a.q, a.q_rows, a.hq, a.q_stride, G, 1) ||
      !make_cache_map(&tk, a.kc, a.num_blocks, a.hkv) ||
      !make_cache_map(&tv, a.vc, a.num_blocks, a.hkv))
    return cudaErrorInvalidValue;
  decode_kernel<MT><<<grid, kThreads, Cfg<MT>::kSmem, st>>>(tq, tk, tv, a, ws);
  return cudaGetLastError();
}

}  // namespace

int decode_grid(int group, int sms) {
  (void)group;
  return sms;  // one CTA per SM
}

cudaError_t launch_decode(const AttnArgs& a, const Workspace& ws, int grid, cudaStream_t st) {
  const int G = a.hq / a.hkv;
  return G <= 16 ? launch_mt<1>(a, ws, grid, st) : launch_mt<2>(a, ws, grid, st);
}

}  // namespace pkv
