// Split-KV decode attention over int8 caches (pkv_attention_int8).
//
// What it computes: the decode attention of pkv_decode.cu ("vLLM 推理全流程深度
// 解析", paged_attention_v1 section; "Tour: One forward pass", stop 10) with
// K_j = k_scale * code and V_j = v_scale * code, the int8 KV cache that the
// closing note of the deep dive's paged_attention section names as a decode
// speed-up.  Work units, split-KV partial results and the merge are those of
// the bf16 path (same plan, same merge of the splits).
//
// GB300 design.  A page of one KV head is 4 KB of codes (16 slots x 128 for K,
// the same for V), loaded by TMA into a per-warp ring (one 2 KB box each for
// K and V, 128-byte swizzle).  With half the bytes of a bf16 page per page of
// work, a warp has less time per page to hide its latencies, so a CTA per SM
// runs 12 independent warps of one 16-row query tile each (groups of up to
// 16 heads; groups of 17 to 32 heads take decode_i8_x2_kernel below: 8 warps
// of two tiles, two pages a step).  The codes go from shared memory straight into
// the operand registers of fp16 mma.sync m16n8k16 — no widened copy of the
// page is written back — because every code -127..127 is an fp16 integer:
// the byte, offset by 128, becomes the low mantissa byte of the fp16 number
// 1024 + byte (one byte permute for two codes), so the MMAs see code + 1152.
// The offset leaves the sums exactly:
//   * a score becomes s + 1152 * sum_d q_d, the same constant for every key
//     of a row, which neither the online softmax (differences of scores and
//     maxima) nor the merge of the splits (differences of the maxima of one
//     row) sees — the maximum a split writes carries the constant;
//   * the output sum becomes O + 1152 * L with L = sum_k p_k over the same
//     fp16 probabilities, which one more MMA per page and tile gives (P times
//     a column of ones, fp32 accumulation) and which is also the row sum the
//     output is divided by.
// Two reorderings make each thread's codes
// contiguous in shared memory, so that a page takes eight 16-byte loads per
// thread and no ldmatrix:
//   * S = Q.K^T sums over the 128 dimensions in any order: k-step ks of the
//     MMA takes dimensions 32 * t + 4 * ks .. + 3 from thread column t (the
//     query fragments are loaded in the same order), so a thread reads 32
//     consecutive codes of each of its two keys;
//   * O = P.V may produce the output dimensions in any order: n-tile dn, MMA
//     column c is dimension 16 * c + dn, so a thread reads 16 consecutive
//     codes of each of its four keys and ends up holding 32 consecutive
//     output dimensions of its rows (16-byte output stores).
// The query is multiplied by scale * log2(e) * k_scale before it is rounded
// to fp16, so the scores come out of the MMA in the log2 domain; the
// probabilities (at most 2^8, the rescale threshold) are fp16 too, and
// v_scale is applied to the output.  Keys past a unit's end get probability
// 0 and their codes are finite, so no V masking is needed.
#include <cuda_fp16.h>

#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int kBox8 = kBlockSize * 128;          // 16 slots x 128 codes (2 KB)
constexpr int kStage8 = 2 * kBox8;               // K box | V box
constexpr int kIdRegs8 = kMaxChunk / kBlockSize / 32;
constexpr uint32_t kSignFlip = 0x80808080u;      // int8 -> offset binary (code + 128)
constexpr uint32_t kOnesF16x2 = 0x3C003C00u;     // fp16 pair (1, 1)

// groups of up to 16 heads: one 16-row query tile per warp, 12 warps of 3
// page stages (160 registers)
struct Cfg8 {
  static constexpr int kWarps = 12;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kStages = 3;
  static constexpr int kQHalf = 16 * 128;               // bf16 query rows x one 64-dim half
  static constexpr int kWarpBytes = kStages * kStage8 + 2 * kQHalf;
  static constexpr int kBarsPerWarp = kStages + 1;      // page stages, query
  static constexpr int kOffBar = kWarps * kWarpBytes;
  static constexpr int kOffCtl = kOffBar + kWarps * kBarsPerWarp * 8;
  static constexpr int kSmem = kOffCtl + 16 + 1024;
};
static_assert(Cfg8::kSmem <= 232448, "shared memory per CTA");

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// D += A(16x16, row) * B(16x8, col); fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two codes plus 1152 as an fp16 pair: u holds offset-binary bytes (code +
// 128); sel picks two of them (0x4140: bytes 0, 1; 0x4342: bytes 2, 3) into
// the low mantissa bytes of 0x6400 (fp16 1024), which gives 1024 + 128 +
// code (1025..1279, exact).  The kernels take the offset out of their sums.
__device__ __forceinline__ uint32_t codes_plus_bias_f16x2(uint32_t u, uint32_t sel) {
  return __byte_perm(u, 0x64646464u, sel);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// a bf16 pair times s as an fp16 pair
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w, float s) {
  return pack_f16(__uint_as_float(w << 16) * s, __uint_as_float(w & 0xFFFF0000u) * s);
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__global__ void __launch_bounds__(Cfg8::kThreads, 1)
    decode_i8_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, AttnArgs a, Workspace ws) {
  using C = Cfg8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.hq / a.hkv;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t wbase = sbase + warp * C::kWarpBytes;  // this warp's page stages
  const uint32_t qbuf = wbase + C::kStages * kStage8;     // bf16 query rows (TMA)
  const uint32_t bars = sbase + C::kOffBar + warp * C::kBarsPerWarp * 8;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  const uint32_t q_bar = bars + 8u * C::kStages;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kOffCtl);

  if (lane == 0) {
    for (int s = 0; s <= C::kStages; ++s) mbar_init(bars + 8u * s, 1);
    if (warp == 0) *abort = 0;
    fence_barrier_init();
  }
  // rows past a unit's qn * G query rows hold zeros or an earlier unit's
  // queries; their results are dropped
  for (int i = lane; i < 2 * 16 * 8; i += 32) {
    const int row = (i >> 3) % 16, half = (i >> 3) / 16, c = i & 7;
    if (row >= G)
      *reinterpret_cast<uint4*>(smem + (qbuf - sbase) + half * C::kQHalf + row * 128 + c * 16) =
          make_uint4(0, 0, 0, 0);
  }
  // the set-up above overlaps the plan kernel; the work list is read after it
  grid_dep_wait();
  grid_dep_launch();
  if (ws.hdr->n_dec_units == 0) return;  // a batch without decode work (every CTA agrees)
  __syncthreads();

  const int n_units = ws.hdr->n_dec_units;
  const uint64_t pol = l2_evict_first();  // K/V pages are read once
  const float sl2 = a.scale * kLog2e * a.k_scale;  // folded into the fp16 query
  const float o_scale = a.v_scale;
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t page_cnt = 0;

  for (uint32_t unit_cnt = 0;; ++unit_cnt) {
    int u = 0;
    if (lane == 0) u = atomicAdd(&ws.hdr->dec_counter, 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    if (u >= n_units || *abort) break;
    const DecUnit un = ws.units[u];
    const int ug = un.gq & 0xFFFF;  // KV head
    const int qn = un.gq >> 16;     // query tokens of the request
    const int k0 = un.k0, k1 = un.k1;
    const int p0 = k0 / kBlockSize;
    const int npages = (k1 + kBlockSize - 1) / kBlockSize - p0;
    const int nrows = qn * G;

    int ids[kIdRegs8];
    {
      const int* btrow = a.bt + (int64_t)un.r * a.bt_width + p0;
#pragma unroll
      for (int j = 0; j < kIdRegs8; ++j) {
        const int p = lane + 32 * j;
        int blk = 0;
        if (p < npages) {
          blk = __ldg(btrow + p);
          if (blk < 0 || (int64_t)blk >= a.num_blocks) {
            atomicOr(ws.err, PKV_DEV_ERR_BLOCK_ID);
            blk = 0;
          }
        }
        ids[j] = blk;
      }
    }
    // query rows token * G + head of this KV head, by TMA (two 64-dim halves)
    if (lane == 0) {
      fence_async_smem();  // the previous unit's reads of the buffer are done
      mbar_expect_tx(q_bar, 2 * nrows * 128);
      for (int i = 0; i < qn; ++i) {
        tma_load_3d(qbuf + i * G * 128, &tm_q, q_bar, 0, ug * G, un.q0 + i);
        tma_load_3d(qbuf + C::kQHalf + i * G * 128, &tm_q, q_bar, 64, ug * G, un.q0 + i);
      }
    }
    int vis[2];
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      const int row = gid + hrow * 8;
      const int ti = row < nrows ? row / G : qn - 1;
      vis[hrow] = min(k1, un.ctx + ti + 1);
    }

    auto issue_page = [&](int p) {
      const uint32_t x = page_cnt + p;
      const int s = x % C::kStages;
      int idv = ids[0];
#pragma unroll
      for (int j = 1; j < kIdRegs8; ++j)
        if ((p >> 5) == j) idv = ids[j];
      const int blk = __shfl_sync(0xffffffffu, idv, p & 31);
      if (lane == 0) {
        fence_async_smem();
        const uint32_t st = wbase + s * kStage8;
        mbar_expect_tx(full_bar(s), kStage8);
        tma_load_4d_hint(st, &tm_k, full_bar(s), 0, ug, 0, blk, pol);
        tma_load_4d_hint(st + kBox8, &tm_v, full_bar(s), 0, ug, 0, blk, pol);
      }
    };
    for (int p = 0; p < C::kStages && p < npages; ++p) issue_page(p);
    if (!mbar_wait_warp(q_bar, unit_cnt & 1, abort, ws.err)) break;

    // fp16 query fragments in the permuted k order: k-step ks, registers
    // {a0, a2} of row r hold dimensions 32 * tig + 4 * ks .. + 3
    uint32_t qa[8][4];
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      const int row = gid + hrow * 8;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        // dimensions 32 * tig + 8 * c .. + 7: half tig / 2, 16-byte chunk
        // 4 * (tig % 2) + c of the row
        const uint4 v = lds128(qbuf + (tig >> 1) * C::kQHalf + sw128(row, (tig & 1) * 4 + c));
        qa[2 * c][hrow] = bf16x2_to_f16x2(v.x, sl2);
        qa[2 * c][2 + hrow] = bf16x2_to_f16x2(v.y, sl2);
        qa[2 * c + 1][hrow] = bf16x2_to_f16x2(v.z, sl2);
        qa[2 * c + 1][2 + hrow] = bf16x2_to_f16x2(v.w, sl2);
      }
    }

    // o: the output sums (+ 1152 * L); lsum: L of rows gid (elements 0, 1)
    // and gid + 8 (2, 3)
    float o[16][4], lsum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int dn = 0; dn < 16; ++dn)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[dn][e] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};

    bool ok = true;
    for (int p = 0; p < npages; ++p) {
      const uint32_t x = page_cnt + p;
      const int s = x % C::kStages;
      if (!mbar_wait_warp(full_bar(s), (x / C::kStages) & 1, abort, ws.err)) {
        ok = false;
        break;
      }
      const int pos0 = k0 + p * kBlockSize;
      const uint32_t st = wbase + s * kStage8;
      // K: keys gid and gid + 8, codes 32 * tig .. + 31 (16-byte chunks
      // 2 * tig, 2 * tig + 1); V: keys 2 * tig, + 1, + 8, + 9, codes
      // 16 * gid .. + 15 (chunk gid)
      const uint4 ka0 = lds128(st + sw128(gid, 2 * tig)), kb0 = lds128(st + sw128(gid, 2 * tig + 1));
      const uint4 ka1 = lds128(st + sw128(gid + 8, 2 * tig));
      const uint4 kb1 = lds128(st + sw128(gid + 8, 2 * tig + 1));
      const uint4 vA = lds128(st + kBox8 + sw128(2 * tig, gid));
      const uint4 vB = lds128(st + kBox8 + sw128(2 * tig + 1, gid));
      const uint4 vC = lds128(st + kBox8 + sw128(2 * tig + 8, gid));
      const uint4 vD = lds128(st + kBox8 + sw128(2 * tig + 9, gid));

      // S = Q K^T (log2 domain) for the page's 16 keys (two n-tiles of 8)
      float sacc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t u0 = (ks < 4 ? word_of(ka0, ks) : word_of(kb0, ks - 4)) ^ kSignFlip;
        const uint32_t u1 = (ks < 4 ? word_of(ka1, ks) : word_of(kb1, ks - 4)) ^ kSignFlip;
        const uint32_t b00 = codes_plus_bias_f16x2(u0, 0x4140);
        const uint32_t b01 = codes_plus_bias_f16x2(u0, 0x4342);
        const uint32_t b10 = codes_plus_bias_f16x2(u1, 0x4140);
        const uint32_t b11 = codes_plus_bias_f16x2(u1, 0x4342);
        mma_f16(sacc[0], qa[ks], b00, b01);
        mma_f16(sacc[1], qa[ks], b10, b11);
      }

      // the stage's codes are all in registers: its next page can be on its
      // way (issued here, behind the S MMAs, whose latency hides the branch)
      __syncwarp();
      if (p + C::kStages < npages) issue_page(p + C::kStages);

      // online softmax in the log2 domain, keys >= the row's limit masked;
      // the output is rescaled only when a row's maximum grows by more than 2^8
      uint32_t pa[4];
      {
        float xs[2][4];
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = nt * 8 + tig * 2 + (e & 1);
            xs[nt][e] = pos0 + tok < vis[e >> 1] ? sacc[nt][e] : -INFINITY;
          }
          mx0 = fmaxf(mx0, fmaxf(xs[nt][0], xs[nt][1]));
          mx1 = fmaxf(mx1, fmaxf(xs[nt][2], xs[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const bool up0 = mx0 > m_run[0] + 8.f, up1 = mx1 > m_run[1] + 8.f;
        if (__any_sync(0xffffffffu, up0 || up1)) {
          const float n0 = up0 ? mx0 : m_run[0], n1 = up1 ? mx1 : m_run[1];
          // (a row that did not grow keeps factor 1: its maximum may still be -inf)
          const float al0 = up0 ? fast_exp2(m_run[0] - n0) : 1.f;
          const float al1 = up1 ? fast_exp2(m_run[1] - n1) : 1.f;
          m_run[0] = n0;
          m_run[1] = n1;
          lsum[0] *= al0;
          lsum[1] *= al0;
          lsum[2] *= al1;
          lsum[3] *= al1;
#pragma unroll
          for (int dn = 0; dn < 16; ++dn) {
            o[dn][0] *= al0;
            o[dn][1] *= al0;
            o[dn][2] *= al1;
            o[dn][3] *= al1;
          }
        }
        // a row with no visible key yet keeps m = -inf: use 0 as its reference
        const float c0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
        const float c1 = m_run[1] == -INFINITY ? 0.f : m_run[1];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          xs[nt][0] = fast_exp2(xs[nt][0] - c0);
          xs[nt][1] = fast_exp2(xs[nt][1] - c0);
          xs[nt][2] = fast_exp2(xs[nt][2] - c1);
          xs[nt][3] = fast_exp2(xs[nt][3] - c1);
        }
        pa[0] = pack_f16(xs[0][0], xs[0][1]);
        pa[1] = pack_f16(xs[0][2], xs[0][3]);
        pa[2] = pack_f16(xs[1][0], xs[1][1]);
        pa[3] = pack_f16(xs[1][2], xs[1][3]);
      }

      // O += P V: code word i of the four key rows (dimensions 16 * gid +
      // 4 * i .. + 3) gives n-tiles dn = 4 * i .. + 3; the byte pairs (key
      // 2 * tig, key 2 * tig + 1) and (key 2 * tig + 8, + 9) of a dimension
      // are interleaved first.  L += P times a column of ones.
      mma_f16(lsum, pa, kOnesF16x2, kOnesF16x2);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t wa = word_of(vA, i), wb = word_of(vB, i);
        const uint32_t wc = word_of(vC, i), wd = word_of(vD, i);
        const uint32_t ab_lo = __byte_perm(wa, wb, 0x5140) ^ kSignFlip;
        const uint32_t ab_hi = __byte_perm(wa, wb, 0x7362) ^ kSignFlip;
        const uint32_t cd_lo = __byte_perm(wc, wd, 0x5140) ^ kSignFlip;
        const uint32_t cd_hi = __byte_perm(wc, wd, 0x7362) ^ kSignFlip;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t ab = e < 2 ? ab_lo : ab_hi, cd = e < 2 ? cd_lo : cd_hi;
          const uint32_t sel = (e & 1) ? 0x4342 : 0x4140;
          const uint32_t b0 = codes_plus_bias_f16x2(ab, sel);
          const uint32_t b1 = codes_plus_bias_f16x2(cd, sel);
          mma_f16(o[4 * i + e], pa, b0, b1);
        }
      }
    }
    if (!ok) break;
    page_cnt += npages;

    // finish: output = (O + 1152 L) / L - 1152; the thread holds output
    // dimensions 32 * tig .. + 31 of rows gid and gid + 8 (dimension
    // 32 * tig + j in o[j][0 / 2] for j < 16, o[j - 16][1 / 3] above)
    const float l0 = lsum[0], l1 = lsum[2];
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      const int rw = gid + 8 * hrow;  // row: token * G + head in group
      if (rw >= nrows) continue;
      const int e0 = 2 * hrow;  // o[][e0]: first 16 dimensions, o[][e0 + 1]: the rest
      if (un.nsplit == 1) {
        const float inv = 1.f / (hrow ? l1 : l0);
        uint16_t* orow = a.out + (int64_t)(un.q0 + rw / G) * a.out_stride +
                         (int64_t)(ug * G + rw % G) * kHeadSize + 32 * tig;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
          for (int q4 = 0; q4 < 2; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int j = q4 * 8 + 2 * k;
              w[k] = pack_bf16((o[j][e0 + h2] * inv - 1152.f) * o_scale,
                               (o[j + 1][e0 + h2] * inv - 1152.f) * o_scale);
            }
            *reinterpret_cast<uint4*>(orow + h2 * 16 + q4 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
          }
      } else {
        const float off = 1152.f * (hrow ? l1 : l0);
        float* prow = ws.part_o + ((int64_t)un.part + rw) * kHeadSize + 32 * tig;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int j = q4 * 4;
            *reinterpret_cast<float4*>(prow + h2 * 16 + j) = make_float4(
                (o[j][e0 + h2] - off) * o_scale, (o[j + 1][e0 + h2] - off) * o_scale,
                (o[j + 2][e0 + h2] - off) * o_scale, (o[j + 3][e0 + h2] - off) * o_scale);
          }
        if (tig == 0)
          *reinterpret_cast<float2*>(ws.part_ml + ((int64_t)un.part + rw) * 2) =
              make_float2(m_run[hrow], hrow ? l1 : l0);
      }
    }
  }
}

cudaError_t launch_i8(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st) {
  using C = Cfg8;
  static std::atomic<bool> attr[kMaxAttrDevices];
  if (cudaError_t e = smem_attr_once(decode_i8_kernel, C::kSmem, attr)) return e;
  const int G = a.hq / a.hkv;
  CUtensorMap tq, tk, tv;
  if (!make_rows_map(&tq, a.q, a.q_rows, a.hq, a.q_stride, G, 1) ||
      !make_cache_map_i8(&tk, a.kc, a.num_blocks, a.hkv) ||
      !make_cache_map_i8(&tv, a.vc, a.num_blocks, a.hkv))
    return cudaErrorInvalidValue;
  return launch_dependent(decode_i8_kernel, dim3(sms), dim3(C::kThreads), C::kSmem, st, tq, tk,
                          tv, a, ws);
}

// Groups of 17 to 32 query heads (two 16-row query tiles): each warp takes two
// pages a step — one online-softmax update over 32 keys, the query fragments
// read once per two pages — so the per-step latency chain (the S MMA chain,
// the max exchange, the P.V issue) is paid once per 32 keys.  Two tiles need
// twice the accumulators, so only 8 warps fit, and a page at a time left
// each warp's chain, not HBM, setting the pace.  The query rows arrive by
// TMA in the buffer their fp16 fragments then replace (a warp reads all its
// rows before it writes a fragment), which leaves shared memory for a ring
// of two page-pair stages per warp (each pair on one barrier: one wait and
// one issue a step).
struct CfgX2 {
  static constexpr int kWarps = 8;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kStages = 2;                        // page pairs
  static constexpr int kQHalf = 32 * 128;                  // bf16 rows x one 64-dim half
  static constexpr int kQ = 2 * kQHalf;                    // = 2 tiles x 8 k-steps x 32 lanes x 16 B
  static constexpr int kWarpBytes = kStages * 2 * kStage8 + kQ;
  static constexpr int kBarsPerWarp = kStages + 1;         // page stages, query
  static constexpr int kOffBar = kWarps * kWarpBytes;
  static constexpr int kOffCtl = kOffBar + kWarps * kBarsPerWarp * 8;
  static constexpr int kSmem = kOffCtl + 16 + 1024;
};
static_assert(CfgX2::kSmem <= 232448, "shared memory per CTA");

__global__ void __launch_bounds__(CfgX2::kThreads, 1)
    decode_i8_x2_kernel(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, AttnArgs a, Workspace ws) {
  using C = CfgX2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.hq / a.hkv;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t wbase = sbase + warp * C::kWarpBytes;  // this warp's page stages
  const uint32_t qbuf = wbase + C::kStages * 2 * kStage8; // query rows, then their fragments
  const uint32_t bars = sbase + C::kOffBar + warp * C::kBarsPerWarp * 8;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  const uint32_t q_bar = bars + 8u * C::kStages;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kOffCtl);

  if (lane == 0) {
    for (int s = 0; s <= C::kStages; ++s) mbar_init(bars + 8u * s, 1);
    if (warp == 0) *abort = 0;
    fence_barrier_init();
  }
  // the set-up above overlaps the plan kernel; the work list is read after it
  grid_dep_wait();
  grid_dep_launch();
  if (ws.hdr->n_dec_units == 0) return;  // a batch without decode work (every CTA agrees)
  __syncthreads();

  const int n_units = ws.hdr->n_dec_units;
  const uint64_t pol = l2_evict_first();  // K/V pages are read once
  const float sl2 = a.scale * kLog2e * a.k_scale;  // folded into the fp16 query
  const float o_scale = a.v_scale;
  const int gid = lane >> 2, tig = lane & 3;
  uint32_t pair_cnt = 0;

  for (uint32_t unit_cnt = 0;; ++unit_cnt) {
    int u = 0;
    if (lane == 0) u = atomicAdd(&ws.hdr->dec_counter, 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    if (u >= n_units || *abort) break;
    const DecUnit un = ws.units[u];
    const int ug = un.gq & 0xFFFF;  // KV head
    const int qn = un.gq >> 16;     // query tokens of the request
    const int k0 = un.k0, k1 = un.k1;
    const int p0 = k0 / kBlockSize;
    const int npages = (k1 + kBlockSize - 1) / kBlockSize - p0;
    const int nrows = qn * G;

    int ids[kIdRegs8];
    {
      const int* btrow = a.bt + (int64_t)un.r * a.bt_width + p0;
#pragma unroll
      for (int j = 0; j < kIdRegs8; ++j) {
        const int p = lane + 32 * j;
        int blk = 0;
        if (p < npages) {
          blk = __ldg(btrow + p);
          if (blk < 0 || (int64_t)blk >= a.num_blocks) {
            atomicOr(ws.err, PKV_DEV_ERR_BLOCK_ID);
            blk = 0;
          }
        }
        ids[j] = blk;
      }
    }
    // query rows token * G + head of this KV head, by TMA (two 64-dim halves)
    // into the buffer the previous unit's fragments were read from
    if (lane == 0) {
      fence_async_smem();
      mbar_expect_tx(q_bar, 2 * nrows * 128);
      for (int i = 0; i < qn; ++i) {
        tma_load_3d(qbuf + i * G * 128, &tm_q, q_bar, 0, ug * G, un.q0 + i);
        tma_load_3d(qbuf + C::kQHalf + i * G * 128, &tm_q, q_bar, 64, ug * G, un.q0 + i);
      }
    }
    int vis[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
      for (int hrow = 0; hrow < 2; ++hrow) {
        const int row = mt * 16 + gid + hrow * 8;
        const int ti = row < nrows ? row / G : qn - 1;
        vis[mt][hrow] = min(k1, un.ctx + ti + 1);
      }

    const int nsteps = (npages + 1) / 2;
    // pages 2 * j and 2 * j + 1 (if any) into pair stage (pair_cnt + j) % kStages
    auto issue_pair = [&](int j) {
      const uint32_t x = pair_cnt + j;
      const int s = x % C::kStages;
      const int pa_ = 2 * j;  // both pages' ids sit in the same register
      int idv = ids[0];
#pragma unroll
      for (int r = 1; r < kIdRegs8; ++r)
        if ((pa_ >> 5) == r) idv = ids[r];
      const int blk0 = __shfl_sync(0xffffffffu, idv, pa_ & 31);
      const int blk1 = __shfl_sync(0xffffffffu, idv, (pa_ + 1) & 31);
      if (lane == 0) {
        const bool two = pa_ + 1 < npages;
        fence_async_smem();
        const uint32_t st = wbase + s * 2 * kStage8;
        mbar_expect_tx(full_bar(s), two ? 2 * kStage8 : kStage8);
        tma_load_4d_hint(st, &tm_k, full_bar(s), 0, ug, 0, blk0, pol);
        tma_load_4d_hint(st + kBox8, &tm_v, full_bar(s), 0, ug, 0, blk0, pol);
        if (two) {
          tma_load_4d_hint(st + kStage8, &tm_k, full_bar(s), 0, ug, 0, blk1, pol);
          tma_load_4d_hint(st + kStage8 + kBox8, &tm_v, full_bar(s), 0, ug, 0, blk1, pol);
        }
      }
    };
    for (int j = 0; j < C::kStages && j < nsteps; ++j) issue_pair(j);
    if (!mbar_wait_warp(q_bar, unit_cnt & 1, abort, ws.err)) break;

    // fp16 query fragments in the permuted k order (k-step ks, registers
    // {a0, a2} of row r hold dimensions 32 * tig + 4 * ks .. + 3), written
    // over the rows once every lane holds its own; rows past nrows are zero
    {
      uint4 raw[2][2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int hrow = 0; hrow < 2; ++hrow) {
          const int row = mt * 16 + gid + hrow * 8;
#pragma unroll
          for (int c = 0; c < 4; ++c)
            raw[mt][hrow][c] = row < nrows ? lds128(qbuf + (tig >> 1) * C::kQHalf +
                                                    sw128(row, (tig & 1) * 4 + c))
                                           : make_uint4(0, 0, 0, 0);
        }
      __syncwarp();
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v0 = raw[mt][0][c], v1 = raw[mt][1][c];
          // k-steps 2c (words x, y) and 2c + 1 (words z, w); rows gid, gid + 8
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(
                           qbuf + ((mt * 8 + 2 * c) * 32 + lane) * 16),
                       "r"(bf16x2_to_f16x2(v0.x, sl2)), "r"(bf16x2_to_f16x2(v1.x, sl2)),
                       "r"(bf16x2_to_f16x2(v0.y, sl2)), "r"(bf16x2_to_f16x2(v1.y, sl2))
                       : "memory");
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(
                           qbuf + ((mt * 8 + 2 * c + 1) * 32 + lane) * 16),
                       "r"(bf16x2_to_f16x2(v0.z, sl2)), "r"(bf16x2_to_f16x2(v1.z, sl2)),
                       "r"(bf16x2_to_f16x2(v0.w, sl2)), "r"(bf16x2_to_f16x2(v1.w, sl2))
                       : "memory");
        }
      __syncwarp();
    }

    // o: the output sums (+ 1152 * L); lsum: L of rows gid (elements 0, 1)
    // and gid + 8 (2, 3)
    float o[2][16][4], lsum[2][4];
    float m_run[2][2];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
      for (int dn = 0; dn < 16; ++dn)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][dn][e] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) lsum[mt][e] = 0.f;
      m_run[mt][0] = m_run[mt][1] = -INFINITY;
    }

    bool ok = true;
    for (int j = 0; j < nsteps; ++j) {
      const int p = 2 * j;
      const bool two = p + 1 < npages;
      const uint32_t xs_ = pair_cnt + j;
      const int s = xs_ % C::kStages;
      if (!mbar_wait_warp(full_bar(s), (xs_ / C::kStages) & 1, abort, ws.err)) {
        ok = false;
        break;
      }
      const int pos0 = k0 + p * kBlockSize;
      // without a second page, the first one's codes stand in for it (finite;
      // its keys lie past the unit's end and are masked)
      const uint32_t st[2] = {wbase + s * 2 * kStage8, wbase + s * 2 * kStage8 + (two ? kStage8 : 0)};

      // S = Q K^T (log2 domain) for the 32 keys: n-tiles 2 * pg + nt hold
      // keys nt * 8 + 0..7 of page pg
      float sacc[2][4][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[mt][nt][e] = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        // K: keys gid and gid + 8 of each page, codes 32 * tig + 16 * half .. + 15
        uint4 kc[2][2];
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
          kc[pg][0] = lds128(st[pg] + sw128(gid, 2 * tig + half));
          kc[pg][1] = lds128(st[pg] + sw128(gid + 8, 2 * tig + half));
        }
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int ks = 4 * half + k4;
          uint32_t qf[2][4];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            const uint4 v = lds128(qbuf + ((mt * 8 + ks) * 32 + lane) * 16);
            qf[mt][0] = v.x;
            qf[mt][1] = v.y;
            qf[mt][2] = v.z;
            qf[mt][3] = v.w;
          }
#pragma unroll
          for (int pg = 0; pg < 2; ++pg) {
            const uint32_t u0 = word_of(kc[pg][0], k4) ^ kSignFlip;
            const uint32_t u1 = word_of(kc[pg][1], k4) ^ kSignFlip;
            const uint32_t b00 = codes_plus_bias_f16x2(u0, 0x4140);
            const uint32_t b01 = codes_plus_bias_f16x2(u0, 0x4342);
            const uint32_t b10 = codes_plus_bias_f16x2(u1, 0x4140);
            const uint32_t b11 = codes_plus_bias_f16x2(u1, 0x4342);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              mma_f16(sacc[mt][2 * pg], qf[mt], b00, b01);
              mma_f16(sacc[mt][2 * pg + 1], qf[mt], b10, b11);
            }
          }
        }
      }
      // V: keys 2 * tig, + 1, + 8, + 9 of each page, codes 16 * gid .. + 15;
      // then the pair stage is free for the pair kStages ahead
      uint4 vc[2][4];
#pragma unroll
      for (int pg = 0; pg < 2; ++pg) {
        vc[pg][0] = lds128(st[pg] + kBox8 + sw128(2 * tig, gid));
        vc[pg][1] = lds128(st[pg] + kBox8 + sw128(2 * tig + 1, gid));
        vc[pg][2] = lds128(st[pg] + kBox8 + sw128(2 * tig + 8, gid));
        vc[pg][3] = lds128(st[pg] + kBox8 + sw128(2 * tig + 9, gid));
      }
      __syncwarp();
      if (j + C::kStages < nsteps) issue_pair(j + C::kStages);

      // online softmax over the 32 keys in the log2 domain, keys >= the
      // row's limit masked; the output is rescaled only when a row's maximum
      // grows by more than 2^8
      uint32_t pa[2][2][4];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        float xs[4][4];
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = nt * 8 + tig * 2 + (e & 1);
            xs[nt][e] = pos0 + tok < vis[mt][e >> 1] ? sacc[mt][nt][e] : -INFINITY;
          }
          mx0 = max3f(mx0, xs[nt][0], xs[nt][1]);
          mx1 = max3f(mx1, xs[nt][2], xs[nt][3]);
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const bool up0 = mx0 > m_run[mt][0] + 8.f, up1 = mx1 > m_run[mt][1] + 8.f;
        if (__any_sync(0xffffffffu, up0 || up1)) {
          const float n0 = up0 ? mx0 : m_run[mt][0], n1 = up1 ? mx1 : m_run[mt][1];
          // (a row that did not grow keeps factor 1: its maximum may still be -inf)
          const float al0 = up0 ? fast_exp2(m_run[mt][0] - n0) : 1.f;
          const float al1 = up1 ? fast_exp2(m_run[mt][1] - n1) : 1.f;
          m_run[mt][0] = n0;
          m_run[mt][1] = n1;
          lsum[mt][0] *= al0;
          lsum[mt][1] *= al0;
          lsum[mt][2] *= al1;
          lsum[mt][3] *= al1;
#pragma unroll
          for (int dn = 0; dn < 16; ++dn) {
            o[mt][dn][0] *= al0;
            o[mt][dn][1] *= al0;
            o[mt][dn][2] *= al1;
            o[mt][dn][3] *= al1;
          }
        }
        // a row with no visible key yet keeps m = -inf: use 0 as its reference
        const float c0 = m_run[mt][0] == -INFINITY ? 0.f : m_run[mt][0];
        const float c1 = m_run[mt][1] == -INFINITY ? 0.f : m_run[mt][1];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          xs[nt][0] = fast_exp2(xs[nt][0] - c0);
          xs[nt][1] = fast_exp2(xs[nt][1] - c0);
          xs[nt][2] = fast_exp2(xs[nt][2] - c1);
          xs[nt][3] = fast_exp2(xs[nt][3] - c1);
        }
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
          pa[mt][pg][0] = pack_f16(xs[2 * pg][0], xs[2 * pg][1]);
          pa[mt][pg][1] = pack_f16(xs[2 * pg][2], xs[2 * pg][3]);
          pa[mt][pg][2] = pack_f16(xs[2 * pg + 1][0], xs[2 * pg + 1][1]);
          pa[mt][pg][3] = pack_f16(xs[2 * pg + 1][2], xs[2 * pg + 1][3]);
        }
      }

      // O += P V, one k-step of 16 keys per page: code word i of the four
      // key rows (dimensions 16 * gid + 4 * i .. + 3) gives n-tiles
      // dn = 4 * i .. + 3; the byte pairs (key 2 * tig, key 2 * tig + 1) and
      // (key 2 * tig + 8, + 9) of a dimension are interleaved first.  L +=
      // P times a column of ones.
#pragma unroll
      for (int pg = 0; pg < 2; ++pg) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) mma_f16(lsum[mt], pa[mt][pg], kOnesF16x2, kOnesF16x2);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t wa = word_of(vc[pg][0], i), wb = word_of(vc[pg][1], i);
          const uint32_t wc = word_of(vc[pg][2], i), wd = word_of(vc[pg][3], i);
          const uint32_t ab_lo = __byte_perm(wa, wb, 0x5140) ^ kSignFlip;
          const uint32_t ab_hi = __byte_perm(wa, wb, 0x7362) ^ kSignFlip;
          const uint32_t cd_lo = __byte_perm(wc, wd, 0x5140) ^ kSignFlip;
          const uint32_t cd_hi = __byte_perm(wc, wd, 0x7362) ^ kSignFlip;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t ab = e < 2 ? ab_lo : ab_hi, cd = e < 2 ? cd_lo : cd_hi;
            const uint32_t sel = (e & 1) ? 0x4342 : 0x4140;
            const uint32_t b0 = codes_plus_bias_f16x2(ab, sel);
            const uint32_t b1 = codes_plus_bias_f16x2(cd, sel);
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) mma_f16(o[mt][4 * i + e], pa[mt][pg], b0, b1);
          }
        }
      }
    }
    if (!ok) break;
    pair_cnt += nsteps;

    // finish: output = (O + 1152 L) / L - 1152; the thread holds output
    // dimensions 32 * tig .. + 31 of rows ra and rb (dimension 32 * tig + j
    // in o[j][0 / 2] for j < 16, o[j - 16][1 / 3] above)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      const float l0 = lsum[mt][0], l1 = lsum[mt][2];
      const int ra = mt * 16 + gid, rb = ra + 8;  // rows: token * G + head in group
#pragma unroll
      for (int hrow = 0; hrow < 2; ++hrow) {
        const int rw = hrow ? rb : ra;
        if (rw >= nrows) continue;
        const int e0 = 2 * hrow;  // o[][e0]: first 16 dimensions, o[][e0 + 1]: the rest
        const float l = hrow ? l1 : l0;
        if (un.nsplit == 1) {
          const float inv = 1.f / l;
          uint16_t* orow = a.out + (int64_t)(un.q0 + rw / G) * a.out_stride +
                           (int64_t)(ug * G + rw % G) * kHeadSize + 32 * tig;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int q4 = 0; q4 < 2; ++q4) {
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int j = q4 * 8 + 2 * k;
                w[k] = pack_bf16((o[mt][j][e0 + h2] * inv - 1152.f) * o_scale,
                                 (o[mt][j + 1][e0 + h2] * inv - 1152.f) * o_scale);
              }
              *reinterpret_cast<uint4*>(orow + h2 * 16 + q4 * 8) = make_uint4(w[0], w[1], w[2], w[3]);
            }
        } else {
          const float off = 1152.f * l;
          float* prow = ws.part_o + ((int64_t)un.part + rw) * kHeadSize + 32 * tig;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              const int j = q4 * 4;
              *reinterpret_cast<float4*>(prow + h2 * 16 + j) = make_float4(
                  (o[mt][j][e0 + h2] - off) * o_scale, (o[mt][j + 1][e0 + h2] - off) * o_scale,
                  (o[mt][j + 2][e0 + h2] - off) * o_scale, (o[mt][j + 3][e0 + h2] - off) * o_scale);
            }
          if (tig == 0)
            *reinterpret_cast<float2*>(ws.part_ml + ((int64_t)un.part + rw) * 2) =
                make_float2(m_run[mt][hrow], hrow ? l1 : l0);
        }
      }
    }
  }
}

cudaError_t launch_i8_x2(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st) {
  using C = CfgX2;
  static std::atomic<bool> attr[kMaxAttrDevices];
  if (cudaError_t e = smem_attr_once(decode_i8_x2_kernel, C::kSmem, attr)) return e;
  const int G = a.hq / a.hkv;
  CUtensorMap tq, tk, tv;
  if (!make_rows_map(&tq, a.q, a.q_rows, a.hq, a.q_stride, G, 1) ||
      !make_cache_map_i8(&tk, a.kc, a.num_blocks, a.hkv) ||
      !make_cache_map_i8(&tv, a.vc, a.num_blocks, a.hkv))
    return cudaErrorInvalidValue;
  return launch_dependent(decode_i8_x2_kernel, dim3(sms), dim3(C::kThreads), C::kSmem, st, tq,
                          tk, tv, a, ws);
}

}  // namespace

int decode_i8_warps(int group) { return group <= 16 ? Cfg8::kWarps : CfgX2::kWarps; }

cudaError_t launch_decode_i8(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st) {
  const int G = a.hq / a.hkv;
  return G <= 16 ? launch_i8(a, ws, sms, st) : launch_i8_x2(a, ws, sms, st);
}

}  // namespace pkv
