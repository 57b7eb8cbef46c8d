// Split-KV decode attention over the paged cache (requests with one query
// token, or a few: speculative or multi-token decode), and the merge of
// split results.
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
// GB300 design.  Decode is bound by HBM: each K/V row is read once per KV head
// and used by the G query heads of that head.
//   * Work unit = (request, KV head, range of at most 2048 keys), listed by the
//     plan kernel.  A CTA per SM holds 8 warps.  Each warp takes units from an
//     atomic cursor and streams the unit's pages by itself: TMA boxes of 16
//     slots x 64 dims (K and V, two halves, 128-byte swizzle) into its own
//     ring of 8 KB page stages, 3 deep.  Warps never wait for each other, so
//     each SM keeps 8 independent streams of loads in flight and 8 warps to
//     hide the latency of the math.
//   * A warp owns the query rows of its KV head in one 16-row tile: row =
//     token * G + head in group, for the request's qn tokens (qn * G at most
//     16; longer requests go to prefill).  Groups above 16 heads (up to 32
//     rows, a single token) run decode_pair_kernel below: a warp pair per
//     unit, one tile per warp, one ring of two-page stages per pair, two
//     pages (32 keys) a step.
//     Row (token i) sees the keys before position ctx + i + 1, ctx = keys
//     before the request's first query token (causal mask inside the
//     request's own tokens).  S = Q.K^T and O += P.V run
//     on the tensor cores with bf16 mma.sync m16n8k16 and fp32 accumulation
//     (with up to 32 heads per K/V row the FMA pipes could not keep pace with
//     HBM); the softmax state stays in registers, row reductions by quad
//     shuffles, exp2 with the scale folded in, and the output is rescaled only
//     when a row's maximum grows by more than 2^8 (exact; rarely needed).
//     Keys past the unit's end are masked in S and their V values zeroed in
//     the fragments, so stale or NaN cache slots never reach the product.
//   * A unit that covers a whole request writes the bf16 output; one split of
//     several writes (max, sum, unnormalised output) in fp32 to the workspace,
//     and the merge of the splits (pkv_combine.cuh) runs afterwards: at the
//     end of the prefill kernel's launch for bf16 calls, in the combine
//     kernel below for int8 calls.  Every mbarrier wait is bounded.
// The int8-cache variant of the decode kernel is in pkv_decode_i8.cu; it
// shares the plan, the work units and the merge.
#include "pkv_combine.cuh"
#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int kCombineThreads = 128;  // merge kernel: 4 warps, one split pair row each
constexpr int kBox = kBlockSize * 128;     // one TMA box: 16 slots x 64 dims (2 KB)
constexpr int kPage = 4 * kBox;            // K lo | K hi | V lo | V hi
constexpr int kIdRegs = kMaxChunk / kBlockSize / 32;  // block ids per lane per unit

// decode_kernel: one 16-row query tile per warp (groups of up to 16 heads;
// larger groups take the warp pairs of decode_pair_kernel)
struct Cfg {
  static constexpr int kWarps = 8;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kStages = 3;
  static constexpr int kStageBytes = kPage;
  static constexpr int kQHalf = 16 * 128;             // query rows x one 64-dim half
  static constexpr int kWarpBytes = kStages * kStageBytes + 2 * kQHalf;
  static constexpr int kBarsPerWarp = kStages + 1;     // page stages, query
  static constexpr int kOffBar = kWarps * kWarpBytes;
  static constexpr int kOffCtl = kOffBar + kWarps * kBarsPerWarp * 8;
  static constexpr int kSmem = kOffCtl + 16 + 1024;
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
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Whether this CTA leaves its SM to the prefill grid, launched after this
// one as its programmatic dependent: when the step has prefill items, the
// first P CTAs of the decode grid exit at once, so that the prefill items
// run on their SMs beside the decode units on the others (the prefill kernel
// does not wait for this grid before its items).  P is the number of SMs on
// which the prefill's key-tile steps (items x tiles) fit into the longest
// item's chain, at most one per item and half of the SMs: fewer would
// lengthen the prefill, more would take SMs the decode units need and sit
// idle once the items are done.  When the decode units fill fewer CTAs than
// the grid has (units_per_cta at a time each), the spare SMs would idle
// anyway: P then grows up to one per item (still at most half of the SMs).
// Every CTA computes the same from the plan header (read after the plan
// wait).
__device__ __forceinline__ bool leaves_sm_to_prefill(const AttnArgs& a, const Workspace& ws,
                                                     int units_per_cta) {
  const int G = a.hq / a.hkv;
  const int per_entry = G % 2 == 0 ? a.hq / 2 : a.hq;  // items (query head pairs) per entry
  const int items = ws.hdr->n_pre_entries * per_entry;
  if (items == 0) return false;
  const long long steps = (long long)ws.hdr->pre_tiles * per_entry;
  const int longest = max(ws.hdr->pre_max_tiles, 1);
  const int cap = min(items, (int)gridDim.x / 2);
  int p = (int)min((long long)cap, (steps + longest - 1) / longest);
  const int spare = (int)gridDim.x - (ws.hdr->n_dec_units + units_per_cta - 1) / units_per_cta;
  if (spare > p) p = min(cap, spare);
  return (int)blockIdx.x < max(p, 1);
}

// a work unit written by the plan kernel
__device__ __forceinline__ DecUnit load_unit(const DecUnit* p) {
  const int4 w0 = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 w1 = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  return DecUnit{w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
}

// keep the bf16 halves of a register whose key index is below `valid`
__device__ __forceinline__ uint32_t mask_pair(uint32_t v, int tok_lo, int valid) {
  const uint32_t lo = tok_lo < valid ? 0x0000FFFFu : 0u;
  const uint32_t hi = tok_lo + 1 < valid ? 0xFFFF0000u : 0u;
  return v & (lo | hi);
}

__global__ void __launch_bounds__(Cfg::kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, AttnArgs a, Workspace ws) {
  using C = Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.hq / a.hkv;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t wbase = sbase + warp * C::kWarpBytes;        // this warp's page stages
  const uint32_t qbuf = wbase + C::kStages * C::kStageBytes;  // and query rows
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
  if (leaves_sm_to_prefill(a, ws, C::kWarps) || ws.hdr->n_dec_units == 0) return;
  __syncthreads();

  const int n_units = ws.hdr->n_dec_units;
  const uint64_t pol = l2_evict_first();  // K/V pages are read once
  const float sl2 = a.scale * kLog2e;
  const int gid = lane >> 2, tig = lane & 3;
  const int mi = lane >> 3, rr = lane & 7;
  uint32_t page_cnt = 0;

  for (uint32_t unit_cnt = 0;; ++unit_cnt) {
    int u = 0;
    if (lane == 0) u = atomicAdd(&ws.hdr->dec_counter, 1);
    u = __shfl_sync(0xffffffffu, u, 0);
    if (u >= n_units || *abort) break;
    const DecUnit un = load_unit(ws.units + u);
    const int ug = un.gq & 0xFFFF;  // KV head
    const int uqn = un.gq >> 16;    // query tokens of the request
    const int k0 = un.k0, k1 = un.k1;
    const int p0 = k0 / kBlockSize;
    const int npages = (k1 + kBlockSize - 1) / kBlockSize - p0;

    // block ids of the unit, one per lane per 32 pages
    int ids[kIdRegs];
    {
      const int* btrow = a.bt + (int64_t)un.r * a.bt_width + p0;
#pragma unroll
      for (int j = 0; j < kIdRegs; ++j) {
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
    // the query rows of this KV head by TMA: for each of the unit's qn query
    // tokens, its G heads (g*G ..), at rows token * G .. token * G + G - 1
    const int qn = uqn, nrows = qn * G;
    if (lane == 0) {
      fence_async_smem();  // the previous unit's reads of the buffer are done
      mbar_expect_tx(q_bar, 2 * nrows * 128);
      const int q0 = un.q0;
      for (int i = 0; i < qn; ++i) {
        tma_load_3d(qbuf + i * G * 128, &tm_q, q_bar, 0, ug * G, q0 + i);
        tma_load_3d(qbuf + C::kQHalf + i * G * 128, &tm_q, q_bar, 64, ug * G, q0 + i);
      }
    }
    // last visible key + 1 of the two rows this thread holds: row (token i,
    // head) sees keys < ctx + i + 1, clipped to the unit
    int vis[2];
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
      const int row = (lane >> 2) + hrow * 8;
      const int ti = row < nrows ? row / G : qn - 1;
      vis[hrow] = min(k1, un.ctx + ti + 1);
    }

    // page p of the unit into stage (page_cnt + p) % kStages; the stage's
    // previous page was consumed by this warp already (program order)
    auto issue_page = [&](int p) {
      const uint32_t x = page_cnt + p;
      const int s = x % C::kStages;
      int idv = ids[0];
#pragma unroll
      for (int j = 1; j < kIdRegs; ++j)
        if ((p >> 5) == j) idv = ids[j];
      const int blk = __shfl_sync(0xffffffffu, idv, p & 31);
      if (lane == 0) {
        fence_async_smem();
        const uint32_t st = wbase + s * C::kStageBytes;
        mbar_expect_tx(full_bar(s), C::kStageBytes);
        tma_load_4d_hint(st, &tm_k, full_bar(s), 0, ug, 0, blk, pol);
        tma_load_4d_hint(st + kBox, &tm_k, full_bar(s), 64, ug, 0, blk, pol);
        tma_load_4d_hint(st + 2 * kBox, &tm_v, full_bar(s), 0, ug, 0, blk, pol);
        tma_load_4d_hint(st + 3 * kBox, &tm_v, full_bar(s), 64, ug, 0, blk, pol);
      }
    };
    for (int p = 0; p < C::kStages && p < npages; ++p) issue_page(p);
    if (!mbar_wait_warp(q_bar, unit_cnt & 1, abort, ws.err)) break;

    // the query fragments, in registers for the whole unit
    uint32_t qa[8][4];
#pragma unroll
    for (int kstep = 0; kstep < 8; ++kstep)
      ldsm_x4(qbuf + (kstep >> 2) * C::kQHalf + sw128(rr + ((mi & 1) << 3),
                                                       (kstep & 3) * 2 + (mi >> 1)),
              qa[kstep][0], qa[kstep][1], qa[kstep][2], qa[kstep][3]);

    float o[16][4];
#pragma unroll
    for (int dn = 0; dn < 16; ++dn)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[dn][e] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    bool ok = true;
    for (int p = 0; p < npages; ++p) {
      const uint32_t x = page_cnt + p;
      const int s = x % C::kStages;
      if (!mbar_wait_warp(full_bar(s), (x / C::kStages) & 1, abort, ws.err)) {
        ok = false;
        break;
      }
      const int pos0 = k0 + p * kBlockSize;
      const int valid = k1 - pos0;  // keys of this page inside the unit
      const uint32_t st = wbase + s * C::kStageBytes;

      // S = Q K^T for the page's 16 keys (two n-tiles of 8)
      float sacc[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
      for (int kstep = 0; kstep < 8; ++kstep) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(st + (kstep >> 2) * kBox + sw128(rr + ((mi >> 1) << 3), (kstep & 3) * 2 + (mi & 1)),
                b0, b1, b2, b3);
        mma_bf16(sacc[0], qa[kstep], b0, b1);
        mma_bf16(sacc[1], qa[kstep], b2, b3);
      }

      // online softmax in the log2 domain, keys >= k1 masked; the output is
      // rescaled only when a row's maximum grows by more than 2^8
      uint32_t pa[4];
      {
        float xs[2][4];
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = nt * 8 + tig * 2 + (e & 1);
            xs[nt][e] = pos0 + tok < vis[e >> 1] ? sacc[nt][e] * sl2 : -INFINITY;
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
          l_run[0] *= al0;
          l_run[1] *= al1;
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
          l_run[0] += xs[nt][0] + xs[nt][1];
          l_run[1] += xs[nt][2] + xs[nt][3];
        }
        pa[0] = pack_bf16(xs[0][0], xs[0][1]);
        pa[1] = pack_bf16(xs[0][2], xs[0][3]);
        pa[2] = pack_bf16(xs[1][0], xs[1][1]);
        pa[3] = pack_bf16(xs[1][2], xs[1][3]);
      }

      // O += P V (V rows read transposed); V of keys past the unit zeroed
#pragma unroll
      for (int dn = 0; dn < 16; dn += 2) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(st + (2 + (dn >> 3)) * kBox + sw128(rr + ((mi & 1) << 3), (dn & 7) + (mi >> 1)),
                  b0, b1, b2, b3);
        if (valid < 16) {
          b0 = mask_pair(b0, 2 * tig, valid);
          b2 = mask_pair(b2, 2 * tig, valid);
          b1 = mask_pair(b1, 8 + 2 * tig, valid);
          b3 = mask_pair(b3, 8 + 2 * tig, valid);
        }
        mma_bf16(o[dn], pa, b0, b1);
        mma_bf16(o[dn + 1], pa, b2, b3);
      }
      __syncwarp();
      if (p + C::kStages < npages) issue_page(p + C::kStages);
    }
    if (!ok) break;
    page_cnt += npages;

    // finish: row sums across the quad, then output or split partials
    float l0 = l_run[0], l1 = l_run[1];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const int ra = gid, rb = ra + 8;  // rows: token * G + head in group
    if (un.nsplit == 1) {
      const int q0 = un.q0;
      // row -> out[q0 + row / G][g * G + row % G]
      uint16_t* oa = a.out + (int64_t)(q0 + ra / G) * a.out_stride +
                     (int64_t)(ug * G + ra % G) * kHeadSize;
      uint16_t* ob = a.out + (int64_t)(q0 + rb / G) * a.out_stride +
                     (int64_t)(ug * G + rb % G) * kHeadSize;
      const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {
        const int col = dn * 8 + tig * 2;
        if (ra < nrows)
          *reinterpret_cast<uint32_t*>(oa + col) = pack_bf16(o[dn][0] * i0, o[dn][1] * i0);
        if (rb < nrows)
          *reinterpret_cast<uint32_t*>(ob + col) = pack_bf16(o[dn][2] * i1, o[dn][3] * i1);
      }
    } else {
      const int64_t pra = (int64_t)un.part + ra, prb = (int64_t)un.part + rb;
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {
        const int col = dn * 8 + tig * 2;
        if (ra < nrows)
          *reinterpret_cast<float2*>(ws.part_o + pra * kHeadSize + col) =
              make_float2(o[dn][0], o[dn][1]);
        if (rb < nrows)
          *reinterpret_cast<float2*>(ws.part_o + prb * kHeadSize + col) =
              make_float2(o[dn][2], o[dn][3]);
      }
      if (tig == 0) {
        if (ra < nrows)
          *reinterpret_cast<float2*>(ws.part_ml + pra * 2) = make_float2(m_run[0], l0);
        if (rb < nrows)
          *reinterpret_cast<float2*>(ws.part_ml + prb * 2) = make_float2(m_run[1], l1);
      }
    }
  }
}

// Groups above 16 heads: a unit's rows are the G heads of its one query token
// (qn * G <= 32 leaves a single token), two 16-row tiles.  A warp pair takes
// the unit: each warp runs one tile's MMA chain, and the two share the unit's
// page ring, so a page is loaded once for both tiles and each warp's chain
// per page is that of a one-tile unit.  The first warp of the pair takes the
// unit from the cursor (and hands it over through shared memory), loads the
// pages, and refills a stage only once both warps have released it.  A step
// takes two pages (32 keys): one online-softmax update and one stage
// hand-over per 32 keys, on a ring of two-page stages.  Each warp reads its
// query fragments from global memory (L2) once per unit, so that shared
// memory holds six pairs' rings.
struct CfgP {
  static constexpr int kPairs = 6;
  static constexpr int kWarps = 2 * kPairs;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kStages = 2;        // two-page stages
  static constexpr int kStage = 2 * kPage;
  static constexpr int kPairBytes = kStages * kStage;
  // per pair: full[kStages], empty[kStages], unit[2]
  static constexpr int kBarsPerPair = 2 * kStages + 2;
  static constexpr int kOffUnit = kPairs * kPairBytes;  // int[kPairs][2]: unit handed over
  static constexpr int kOffBar = kOffUnit + kPairs * 2 * 4;
  static constexpr int kOffCtl = kOffBar + kPairs * kBarsPerPair * 8;
  static constexpr int kSmem = kOffCtl + 16 + 1024;
};
static_assert(CfgP::kSmem <= 232448, "shared memory per CTA");

__global__ void __launch_bounds__(CfgP::kThreads, 1)
    decode_pair_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, AttnArgs a, Workspace ws) {
  using C = CfgP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int pair = warp >> 1, tile = warp & 1;  // tile 0: the pair's first warp
  const int G = a.hq / a.hkv;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t pbase = sbase + pair * C::kPairBytes;  // the pair's page stages
  const uint32_t bars = sbase + C::kOffBar + pair * C::kBarsPerPair * 8;
  auto full_bar = [&](int st) { return bars + 8u * st; };
  auto empty_bar = [&](int st) { return bars + 8u * (C::kStages + st); };
  auto unit_bar = [&](int k) { return bars + 8u * (2 * C::kStages + k); };
  volatile int* uslot = reinterpret_cast<volatile int*>(smem + C::kOffUnit) + 2 * pair;
  volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kOffCtl);

  if (tile == 0) {
    if (lane == 0) {
      for (int st = 0; st < C::kStages; ++st) {
        mbar_init(full_bar(st), 1);
        mbar_init(empty_bar(st), 2);  // both warps release a stage
      }
      mbar_init(unit_bar(0), 1);
      mbar_init(unit_bar(1), 1);
      if (warp == 0) *abort = 0;
      fence_barrier_init();
    }
  }
  // the set-up above overlaps the plan kernel; the work list is read after it
  grid_dep_wait();
  grid_dep_launch();
  if (leaves_sm_to_prefill(a, ws, C::kPairs) || ws.hdr->n_dec_units == 0) return;
  __syncthreads();

  const int n_units = ws.hdr->n_dec_units;
  const uint64_t pol = l2_evict_first();  // K/V pages are read once
  const float sl2 = a.scale * kLog2e;
  const int gid = lane >> 2, tig = lane & 3;
  const int mi = lane >> 3, rr = lane & 7;
  const int roff = 16 * tile;  // this warp's rows (heads of the group)
  uint32_t step_cnt = 0;

  for (uint32_t unit_cnt = 0;; ++unit_cnt) {
    const int slot = unit_cnt & 1;
    int u = 0;
    if (tile == 0) {
      if (lane == 0) {
        u = atomicAdd(&ws.hdr->dec_counter, 1);
        uslot[slot] = u;
        mbar_arrive(unit_bar(slot));
      }
      u = __shfl_sync(0xffffffffu, u, 0);
    } else {
      if (!mbar_wait_warp(unit_bar(slot), (unit_cnt >> 1) & 1, abort, ws.err)) break;
      u = uslot[slot];
    }
    if (u >= n_units || *abort) break;
    const DecUnit un = load_unit(ws.units + u);
    const int ug = un.gq & 0xFFFF;  // KV head
    const int k0 = un.k0, k1 = un.k1;
    const int p0 = k0 / kBlockSize;
    const int npages = (k1 + kBlockSize - 1) / kBlockSize - p0;
    const int nrows = G;            // one query token: the group's heads

    // block ids of the unit (the loading warp only), one per lane per 32 pages
    int ids[kIdRegs];
#pragma unroll
    for (int j = 0; j < kIdRegs; ++j) ids[j] = 0;
    if (tile == 0) {
      const int* btrow = a.bt + (int64_t)un.r * a.bt_width + p0;
#pragma unroll
      for (int j = 0; j < kIdRegs; ++j) {
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
    // pages 2 * j and 2 * j + 1 (if any) of the unit into stage
    // (step_cnt + j) % kStages, once both warps have released the stage's
    // previous pages
    const int nsteps = (npages + 1) / 2;
    bool ok = true;
    auto issue_step = [&](int j) {
      const uint32_t x = step_cnt + j;
      const int st = x % C::kStages;
      if (x >= (uint32_t)C::kStages &&
          !mbar_wait_warp(empty_bar(st), ((x / C::kStages) - 1) & 1, abort, ws.err)) {
        ok = false;
        return;
      }
      const int p = 2 * j;  // both pages' ids sit in the same register
      int idv = ids[0];
#pragma unroll
      for (int r = 1; r < kIdRegs; ++r)
        if ((p >> 5) == r) idv = ids[r];
      const int blk0 = __shfl_sync(0xffffffffu, idv, p & 31);
      const int blk1 = __shfl_sync(0xffffffffu, idv, (p + 1) & 31);
      if (lane == 0) {
        const bool two = p + 1 < npages;
        const uint32_t sa = pbase + st * C::kStage;
        mbar_expect_tx(full_bar(st), two ? 2 * kPage : kPage);
        tma_load_4d_hint(sa, &tm_k, full_bar(st), 0, ug, 0, blk0, pol);
        tma_load_4d_hint(sa + kBox, &tm_k, full_bar(st), 64, ug, 0, blk0, pol);
        tma_load_4d_hint(sa + 2 * kBox, &tm_v, full_bar(st), 0, ug, 0, blk0, pol);
        tma_load_4d_hint(sa + 3 * kBox, &tm_v, full_bar(st), 64, ug, 0, blk0, pol);
        if (two) {
          const uint32_t sb = sa + kPage;
          tma_load_4d_hint(sb, &tm_k, full_bar(st), 0, ug, 0, blk1, pol);
          tma_load_4d_hint(sb + kBox, &tm_k, full_bar(st), 64, ug, 0, blk1, pol);
          tma_load_4d_hint(sb + 2 * kBox, &tm_v, full_bar(st), 0, ug, 0, blk1, pol);
          tma_load_4d_hint(sb + 3 * kBox, &tm_v, full_bar(st), 64, ug, 0, blk1, pol);
        }
      }
    };
    if (tile == 0) {
      for (int j = 0; j < C::kStages && j < nsteps && ok; ++j) issue_step(j);
      if (!ok) break;
    }
    // every row sees keys < ctx + 1, clipped to the unit
    const int vis = min(k1, un.ctx + 1);
    // the A fragments of the warp's 16 query rows (heads roff + gid and
    // roff + gid + 8 of the group; k-step k: dimensions 16k + 2tig, + 1 in
    // registers 0 / 1 and 16k + 8 + 2tig, + 1 in 2 / 3); rows past the
    // group's G heads are zero and their results dropped
    uint32_t qa[8][4];
    {
      const int ha = roff + gid, hb = ha + 8;
      const uint16_t* qrow = a.q + (int64_t)un.q0 * a.q_stride + (int64_t)ug * G * kHeadSize;
      const uint32_t* qra = reinterpret_cast<const uint32_t*>(qrow + (int64_t)ha * kHeadSize);
      const uint32_t* qrb = reinterpret_cast<const uint32_t*>(qrow + (int64_t)hb * kHeadSize);
#pragma unroll
      for (int kstep = 0; kstep < 8; ++kstep) {
        qa[kstep][0] = ha < G ? __ldg(qra + 8 * kstep + tig) : 0u;
        qa[kstep][1] = hb < G ? __ldg(qrb + 8 * kstep + tig) : 0u;
        qa[kstep][2] = ha < G ? __ldg(qra + 8 * kstep + 4 + tig) : 0u;
        qa[kstep][3] = hb < G ? __ldg(qrb + 8 * kstep + 4 + tig) : 0u;
      }
    }

    float o[16][4];
#pragma unroll
    for (int dn = 0; dn < 16; ++dn)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[dn][e] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    for (int j = 0; j < nsteps; ++j) {
      const uint32_t x = step_cnt + j;
      const int st = x % C::kStages;
      if (!mbar_wait_warp(full_bar(st), (x / C::kStages) & 1, abort, ws.err)) {
        ok = false;
        break;
      }
      const int p = 2 * j;
      const bool two = p + 1 < npages;
      const int pos0 = k0 + p * kBlockSize;
      // keys of each page inside the unit (a missing second page: none, its
      // keys masked and its V zeroed; the first page's data stands in)
      const int valid[2] = {k1 - pos0, k1 - pos0 - kBlockSize};
      const uint32_t sa[2] = {pbase + st * C::kStage, pbase + st * C::kStage + (two ? kPage : 0)};

      // S = Q K^T for the step's 32 keys (n-tiles 2 * page + 0, 1 of 8 keys)
      float sacc[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
#pragma unroll
      for (int kstep = 0; kstep < 8; ++kstep) {
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sa[pg] + (kstep >> 2) * kBox +
                      sw128(rr + ((mi >> 1) << 3), (kstep & 3) * 2 + (mi & 1)),
                  b0, b1, b2, b3);
          mma_bf16(sacc[2 * pg], qa[kstep], b0, b1);
          mma_bf16(sacc[2 * pg + 1], qa[kstep], b2, b3);
        }
      }

      // online softmax in the log2 domain (as in decode_kernel)
      uint32_t pa[2][4];
      {
        float xs[4][4];
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int tok = nt * 8 + tig * 2 + (e & 1);
            xs[nt][e] = pos0 + tok < vis ? sacc[nt][e] * sl2 : -INFINITY;
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
          const float al0 = up0 ? fast_exp2(m_run[0] - n0) : 1.f;
          const float al1 = up1 ? fast_exp2(m_run[1] - n1) : 1.f;
          m_run[0] = n0;
          m_run[1] = n1;
          l_run[0] *= al0;
          l_run[1] *= al1;
#pragma unroll
          for (int dn = 0; dn < 16; ++dn) {
            o[dn][0] *= al0;
            o[dn][1] *= al0;
            o[dn][2] *= al1;
            o[dn][3] *= al1;
          }
        }
        const float c0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
        const float c1 = m_run[1] == -INFINITY ? 0.f : m_run[1];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
          xs[nt][0] = fast_exp2(xs[nt][0] - c0);
          xs[nt][1] = fast_exp2(xs[nt][1] - c0);
          xs[nt][2] = fast_exp2(xs[nt][2] - c1);
          xs[nt][3] = fast_exp2(xs[nt][3] - c1);
          l_run[0] += xs[nt][0] + xs[nt][1];
          l_run[1] += xs[nt][2] + xs[nt][3];
        }
#pragma unroll
        for (int pg = 0; pg < 2; ++pg) {
          pa[pg][0] = pack_bf16(xs[2 * pg][0], xs[2 * pg][1]);
          pa[pg][1] = pack_bf16(xs[2 * pg][2], xs[2 * pg][3]);
          pa[pg][2] = pack_bf16(xs[2 * pg + 1][0], xs[2 * pg + 1][1]);
          pa[pg][3] = pack_bf16(xs[2 * pg + 1][2], xs[2 * pg + 1][3]);
        }
      }

      // O += P V (V rows read transposed), one k-step of 16 keys per page;
      // V of keys past the unit zeroed
#pragma unroll
      for (int pg = 0; pg < 2; ++pg)
#pragma unroll
        for (int dn = 0; dn < 16; dn += 2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sa[pg] + (2 + (dn >> 3)) * kBox +
                        sw128(rr + ((mi & 1) << 3), (dn & 7) + (mi >> 1)),
                    b0, b1, b2, b3);
          if (valid[pg] < 16) {
            b0 = mask_pair(b0, 2 * tig, valid[pg]);
            b2 = mask_pair(b2, 2 * tig, valid[pg]);
            b1 = mask_pair(b1, 8 + 2 * tig, valid[pg]);
            b3 = mask_pair(b3, 8 + 2 * tig, valid[pg]);
          }
          mma_bf16(o[dn], pa[pg], b0, b1);
          mma_bf16(o[dn + 1], pa[pg], b2, b3);
        }
      // this warp is done with the stage; the loading warp refills it
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(st));
      if (tile == 0 && j + C::kStages < nsteps) {
        issue_step(j + C::kStages);
        if (!ok) break;
      }
    }
    if (!ok) break;
    step_cnt += nsteps;

    // finish: row sums across the quad, then output or split partials
    float l0 = l_run[0], l1 = l_run[1];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const int ra = roff + gid, rb = ra + 8;  // rows: heads of the group
    if (un.nsplit == 1) {
      uint16_t* oa = a.out + (int64_t)un.q0 * a.out_stride + (int64_t)(ug * G + ra) * kHeadSize;
      uint16_t* ob = a.out + (int64_t)un.q0 * a.out_stride + (int64_t)(ug * G + rb) * kHeadSize;
      const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {
        const int col = dn * 8 + tig * 2;
        if (ra < nrows)
          *reinterpret_cast<uint32_t*>(oa + col) = pack_bf16(o[dn][0] * i0, o[dn][1] * i0);
        if (rb < nrows)
          *reinterpret_cast<uint32_t*>(ob + col) = pack_bf16(o[dn][2] * i1, o[dn][3] * i1);
      }
    } else {
      const int64_t pra = (int64_t)un.part + ra, prb = (int64_t)un.part + rb;
#pragma unroll
      for (int dn = 0; dn < 16; ++dn) {
        const int col = dn * 8 + tig * 2;
        if (ra < nrows)
          *reinterpret_cast<float2*>(ws.part_o + pra * kHeadSize + col) =
              make_float2(o[dn][0], o[dn][1]);
        if (rb < nrows)
          *reinterpret_cast<float2*>(ws.part_o + prb * kHeadSize + col) =
              make_float2(o[dn][2], o[dn][3]);
      }
      if (tig == 0) {
        if (ra < nrows)
          *reinterpret_cast<float2*>(ws.part_ml + pra * 2) = make_float2(m_run[0], l0);
        if (rb < nrows)
          *reinterpret_cast<float2*>(ws.part_ml + prb * 2) = make_float2(m_run[1], l1);
      }
    }
  }
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(AttnArgs a, Workspace ws) {
  constexpr int kWarpsPerBlock = kCombineThreads / 32;
  grid_dep_wait();  // the decode kernel's partial results
  combine_splits(a, ws, blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5), gridDim.x * kWarpsPerBlock);
}

cudaError_t launch_one_tile(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st) {
  using C = Cfg;
  static std::atomic<bool> attr[kMaxAttrDevices];
  if (cudaError_t e = smem_attr_once(decode_kernel, C::kSmem, attr)) return e;
  const int G = a.hq / a.hkv;
  CUtensorMap tq, tk, tv;
  if (!make_rows_map(&tq, a.q, a.q_rows, a.hq, a.q_stride, G, 1) ||
      !make_cache_map(&tk, a.kc, a.num_blocks, a.hkv) ||
      !make_cache_map(&tv, a.vc, a.num_blocks, a.hkv))
    return cudaErrorInvalidValue;
  return launch_dependent(decode_kernel, dim3(sms), dim3(C::kThreads), C::kSmem, st, tq, tk,
                          tv, a, ws);
}

cudaError_t launch_pair(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st) {
  static std::atomic<bool> attr[kMaxAttrDevices];
  if (cudaError_t e = smem_attr_once(decode_pair_kernel, CfgP::kSmem, attr)) return e;
  CUtensorMap tk, tv;  // (query rows: plain loads, 16-byte aligned by the API's checks)
  if (!make_cache_map(&tk, a.kc, a.num_blocks, a.hkv) ||
      !make_cache_map(&tv, a.vc, a.num_blocks, a.hkv))
    return cudaErrorInvalidValue;
  return launch_dependent(decode_pair_kernel, dim3(sms), dim3(CfgP::kThreads), CfgP::kSmem, st,
                          tk, tv, a, ws);
}

}  // namespace

int decode_workers(int group, int kv_int8, int sms) {
  return sms * (kv_int8 ? decode_i8_warps(group) : (group <= 16 ? Cfg::kWarps : CfgP::kPairs));
}

cudaError_t launch_decode(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st) {
  const int G = a.hq / a.hkv;
  if (a.kv_int8) return launch_decode_i8(a, ws, sms, st);
  return G <= 16 ? launch_one_tile(a, ws, sms, st) : launch_pair(a, ws, sms, st);
}

cudaError_t launch_combine(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st) {
  return launch_dependent(combine_kernel, dim3(sms * 8), dim3(kCombineThreads), 0, st, a, ws);
}

}  // namespace pkv
