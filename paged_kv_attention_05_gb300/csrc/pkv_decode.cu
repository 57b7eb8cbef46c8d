// Split-KV decode attention over the paged cache (requests with one query
// token), with the split merge fused into the last unit of each
// (request, KV head).
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
// per KV head and used by G query heads.  So
//   * one unit = (request, KV head, key range <= 1024): the G query heads of
//     the KV head are packed as the rows of a 16- or 32-row tile, so each
//     K/V byte is fetched once for all of them;
//   * a persistent grid (SMs x resident CTAs) pulls units from an atomic
//     cursor, so skewed lengths balance without a host-side plan;
//   * K/V tiles of 64 tokens (4 pages, each located through the block table)
//     stream into a 3-stage cp.async ring in shared memory, 16-byte pieces
//     XOR-swizzled by row so that ldmatrix reads are bank-conflict free; rows
//     past the unit's last key are zero-filled, never read;
//   * each warp owns one page of every stage: S = Q.K^T and O += P.V run on
//     the tensor cores with bf16 mma.sync (m16n8k16, fp32 accumulation) —
//     with G up to 32 heads per K/V row the FMA pipes could not keep up with
//     HBM — and the softmax state (running max, sum) lives in registers with
//     quad shuffles for the row reductions (exp2 with the scale folded);
//   * the four warps' partial states merge through shared memory at the end
//     of a unit; a unit that is one of several splits writes (max, sum,
//     unnormalised output) in fp32 to the workspace and takes a ticket; the
//     last split to arrive merges all splits and writes the bf16 output.
//     Nothing ever waits on another CTA.
#include <cuda_bf16.h>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kStageBytes = 2 * kDecTile * kHeadSize * 2;  // K and V of one stage
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

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

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// byte offset of 16-byte piece c of row `row` in a [rows][256 B] swizzled tile
__device__ __forceinline__ uint32_t swz(int row, int c) {
  return (uint32_t)(row * 256 + ((c ^ (row & 7)) << 4));
}

template <int MT>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(AttnArgs a, Workspace ws) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* kv_s = smem;                                  // kDecStages x (K | V)
  uint8_t* q_s = smem + kDecStages * kStageBytes;        // [MT*16][256 B]
  __shared__ int s_unit;
  __shared__ int s_ticket;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = a.hq / a.hkv;
  const float sl2 = a.scale * kLog2e;
  const int64_t row_elems = (int64_t)a.hkv * kHeadSize;  // elements per cache slot
  const int n_units = ws.hdr->n_dec_units;

  for (;;) {
    if (tid == 0) s_unit = atomicAdd(&ws.hdr->dec_counter, 1);
    __syncthreads();
    const int u = s_unit;
    if (u >= n_units) break;
    const DecUnit un = ws.units[u];
    const int r = un.r, g = un.g, k0 = un.k0, k1 = un.k1;
    const int q0 = a.qsl[r];
    const int ntiles = (k1 - k0 + kDecTile - 1) / kDecTile;
    const int* btrow = a.bt + (int64_t)r * a.bt_width;
    const uint16_t* kbase = a.kc + (int64_t)g * kHeadSize;
    const uint16_t* vbase = a.vc + (int64_t)g * kHeadSize;

    // the G query rows of this KV head, zero rows up to MT*16
    for (int i = tid; i < MT * 16 * 16; i += kDecThreads) {
      const int row = i >> 4, c = i & 15;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (row < G)
        val = *reinterpret_cast<const uint4*>(a.q + (int64_t)q0 * a.q_stride +
                                              (int64_t)(g * G + row) * kHeadSize + c * 8);
      *reinterpret_cast<uint4*>(q_s + swz(row, c)) = val;
    }

    auto load_tile = [&](int t, int stage) {
      const int c = tid & 15;
      uint8_t* ks = kv_s + stage * kStageBytes;
      uint8_t* vs = ks + kStageBytes / 2;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = (tid >> 4) + 8 * i;
        const int pos = k0 + t * kDecTile + row;
        int bytes = 0;
        const uint16_t* ksrc = kbase;
        const uint16_t* vsrc = vbase;
        if (pos < k1) {
          const int blk = __ldg(btrow + (pos >> 4));
          if (blk >= 0 && (int64_t)blk < a.num_blocks) {
            const int64_t off = ((int64_t)blk * kBlockSize + (pos & 15)) * row_elems + c * 8;
            ksrc = kbase + off;
            vsrc = vbase + off;
            bytes = 16;
          } else if (c == 0) {
            atomicOr(ws.err, PKV_DEV_ERR_BLOCK_ID);
          }
        }
        cp_async16(smem_u32(ks + swz(row, c)), ksrc, bytes);
        cp_async16(smem_u32(vs + swz(row, c)), vsrc, bytes);
      }
    };

#pragma unroll
    for (int s = 0; s < kDecStages - 1; ++s) {
      if (s < ntiles) load_tile(s, s);
      cp_async_commit();
    }

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

    const int gid = lane >> 2, tig = lane & 3;
    for (int t = 0; t < ntiles; ++t) {
      cp_async_wait<kDecStages - 2>();
      __syncthreads();
      if (t + kDecStages - 1 < ntiles) load_tile(t + kDecStages - 1, (t + kDecStages - 1) % kDecStages);
      cp_async_commit();

      const int pos0 = k0 + t * kDecTile + warp * 16;
      if (pos0 >= k1) continue;  // this warp's page of the last tile is empty
      const uint8_t* ks = kv_s + (t % kDecStages) * kStageBytes + warp * 16 * 256;
      const uint8_t* vs = ks + kStageBytes / 2;

      // S = Q K^T for 16 tokens (two n-tiles of 8)
      float sacc[MT][2][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.f;
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int kstep = 0; kstep < 8; ++kstep) {
        uint32_t b0, b1, b2, b3;
        {
          const int tok = rr + ((mi >> 1) << 3);
          const int ch = kstep * 2 + (mi & 1);
          ldsm_x4(smem_u32(ks) + swz(tok, ch), b0, b1, b2, b3);
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          uint32_t a0, a1, a2, a3;
          const int qrow = mt * 16 + rr + ((mi & 1) << 3);
          const int ch = kstep * 2 + (mi >> 1);
          ldsm_x4(smem_u32(q_s) + swz(qrow, ch), a0, a1, a2, a3);
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
            x[nt][e] = (pos0 + tok < k1) ? sacc[mt][nt][e] * sl2 : -INFINITY;
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

      // O += P V (V rows read transposed)
#pragma unroll
      for (int dn = 0; dn < 16; dn += 2) {
        uint32_t b0, b1, b2, b3;
        const int tok = rr + ((mi & 1) << 3);
        const int ch = dn + (mi >> 1);
        ldsm_x4_t(smem_u32(vs) + swz(tok, ch), b0, b1, b2, b3);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          mma_bf16(o[mt][dn], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b0, b1);
          mma_bf16(o[mt][dn + 1], pa[mt][0], pa[mt][1], pa[mt][2], pa[mt][3], b2, b3);
        }
      }
    }
    cp_async_wait<0>();
    __syncthreads();  // pipeline drained: the stage ring is free for the merge

    // merge the four warps' states: [warp][row] m, l and [warp][row][128] o
    const int ROWS = MT * 16;
    float* mw = reinterpret_cast<float*>(kv_s);
    float* lw = mw + 4 * ROWS;
    float* ow = lw + 4 * ROWS;
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
        float* pa_ = ow + ((int64_t)warp * ROWS + ra) * kHeadSize + col;
        float* pb_ = ow + ((int64_t)warp * ROWS + rb) * kHeadSize + col;
        pa_[0] = o[mt][dn][0];
        pa_[1] = o[mt][dn][1];
        pb_[0] = o[mt][dn][2];
        pb_[1] = o[mt][dn][3];
      }
    }
    __syncthreads();

    const int d = tid;  // one output column per thread
    if (un.nsplit == 1) {
      for (int row = 0; row < G; ++row) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * ROWS + row]);
        float acc = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float f = fast_exp2(mw[w * ROWS + row] - M);
          acc += f * ow[((int64_t)w * ROWS + row) * kHeadSize + d];
          lsum += f * lw[w * ROWS + row];
        }
        a.out[(int64_t)q0 * a.out_stride + (int64_t)(g * G + row) * kHeadSize + d] =
            __bfloat16_as_ushort(__float2bfloat16_rn(acc / lsum));
      }
    } else {
      for (int row = 0; row < G; ++row) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < 4; ++w) M = fmaxf(M, mw[w * ROWS + row]);
        float acc = 0.f, lsum = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float f = fast_exp2(mw[w * ROWS + row] - M);
          acc += f * ow[((int64_t)w * ROWS + row) * kHeadSize + d];
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
      __syncthreads();
      if (tid == 0) s_ticket = atomicAdd(&ws.counters[(int64_t)r * a.hkv + g], 1);
      __syncthreads();
      if (s_ticket == un.nsplit - 1) {
        // last split to finish: merge all splits of (r, g)
        __threadfence();
        const int first = un.part - un.split;
        for (int row = 0; row < G; ++row) {
          float M = -INFINITY;
          for (int s = 0; s < un.nsplit; ++s)
            M = fmaxf(M, __ldcg(ws.part_ml + ((int64_t)(first + s) * G + row) * 2));
          float acc = 0.f, lsum = 0.f;
          for (int s = 0; s < un.nsplit; ++s) {
            const int64_t prow = (int64_t)(first + s) * G + row;
            const float f = fast_exp2(__ldcg(ws.part_ml + prow * 2) - M);
            acc += f * __ldcg(ws.part_o + prow * kHeadSize + d);
            lsum += f * __ldcg(ws.part_ml + prow * 2 + 1);
          }
          a.out[(int64_t)q0 * a.out_stride + (int64_t)(g * G + row) * kHeadSize + d] =
              __bfloat16_as_ushort(__float2bfloat16_rn(acc / lsum));
        }
      }
    }
    __syncthreads();  // merge buffers and s_unit are reused by the next unit
  }
}

template <int MT>
size_t decode_smem() {
  return (size_t)kDecStages * kStageBytes + (size_t)MT * 16 * 256;
}

template <int MT>
int decode_occupancy() {
  static int occ = -1;
  if (occ < 0) {
    cudaFuncSetAttribute(decode_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)decode_smem<MT>());
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<MT>, kDecThreads,
                                                      decode_smem<MT>()) != cudaSuccess)
      n = 1;
    occ = n < 1 ? 1 : n;
  }
  return occ;
}

}  // namespace

int decode_ctas_per_sm(int group) {
  return group <= 16 ? decode_occupancy<1>() : decode_occupancy<2>();
}

cudaError_t launch_decode(const AttnArgs& a, const Workspace& ws, int grid, cudaStream_t st) {
  const int G = a.hq / a.hkv;
  if (G <= 16) {
    decode_occupancy<1>();
    decode_kernel<1><<<grid, kDecThreads, decode_smem<1>(), st>>>(a, ws);
  } else {
    decode_occupancy<2>();
    decode_kernel<2><<<grid, kDecThreads, decode_smem<2>(), st>>>(a, ws);
  }
  return cudaGetLastError();
}

}  // namespace pkv
