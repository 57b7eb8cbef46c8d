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
// GB300 design.  A work item is a 128-row query tile of one request for two
// query heads of the same KV head (one head when Hq / Hkv is odd): tiles "a"
// and "b" share every K/V tile.  A persistent grid (one CTA per SM, all 512
// TMEM columns) takes items from an atomic cursor, longest first.  Roles:
//   warp 0      producer: publishes the item in a two-slot ring, loads the two
//               Q tiles by TMA as soon as the previous item's last S = Q K^T
//               has consumed them, then the K and V tiles of 128 keys (8 pages
//               each, one 16-slot x 64-dim box per page and half, 128-byte
//               swizzle) into a 2-stage ring, K and V released separately; in
//               a request's last tile it zero-fills the V rows of keys past
//               seq_len so that no stale value (NaN) reaches P.V;
//   warp 1      allocates TMEM and issues every MMA from one thread, in the
//               order S_a(0) S_b(0) | PV_a(j) S_a(j+1) PV_b(j) S_b(j+1) ...:
//               S into TMEM, P taken from TMEM (the scores' columns,
//               overwritten with bf16 probabilities) and V from shared memory
//               (MN-major), O accumulating in TMEM; tcgen05.commit drives the
//               mbarriers.  Because one thread's MMAs complete in order, S(j+1)
//               being ready also means PV(j) is done;
//   warps 2-9   softmax, two warps per row quarter (one per 64-key half of
//               the scores), one query row per thread (TMEM lane = 32 *
//               (warp % 4) + lane = row), both query tiles in turn: scores ->
//               causal/length mask (only on tiles that cross the diagonal) ->
//               running max in the log2 domain -> exp2 -> row sum -> bf16 P
//               back into TMEM.  O is rescaled in TMEM only when a row's max
//               grows by more than 2^8 (exact, rare).  At the end of an item
//               each warp leaves its partial row sums in shared memory;
//   warps 10-13 epilogue: once O_x is final, read it out of TMEM in two
//               64-column halves, divide by the row sum, release O_x to the
//               next item's first P.V and write the bf16 rows to global memory
//               through a per-warp staging area (whole 64-byte row pieces).
// Every mbarrier wait is bounded; on expiry the kernel records
// PKV_DEV_ERR_TIMEOUT, stops issuing work, frees its TMEM and returns.
#include "pkv_combine.cuh"
#include "pkv_device.cuh"

namespace pkv {
namespace {

using namespace dev;

constexpr int kThreads = 448;                     // 14 warps
constexpr int kStages = 2;
constexpr int kTileK = 128;                       // keys per KV tile
constexpr int kHalfBytes = 128 * 128;             // 128 rows x 64 bf16
constexpr int kTileBytes = 2 * kHalfBytes;        // a Q, K or V tile: 32 KB
constexpr int kPageBoxBytes = 16 * 128;           // one 16-slot x 64-dim box
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;         // log2 units

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;                          // Q_a | Q_b
constexpr int kOffK = kOffQ + 2 * kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kStageWarp = 32 * 64;               // epilogue staging: 32 rows x 64 bytes
constexpr int kOffStage = kOffV + kStages * kTileBytes;  // one staging area per epilogue warp
constexpr int kOffLsum = kOffStage + 4 * kStageWarp;  // [2 items][2 tiles][2 halves][128 rows]
constexpr int kOffBar = kOffLsum + 2 * 2 * 2 * 128 * 4;
enum {
  B_QF = 0,   // [2] Q tile loaded
  B_QE = 2,   // [2] Q tile consumed by the item's last S
  B_KF = 4,   // [2] K stage loaded
  B_KE = 6,   // [2] K stage free
  B_VF = 8,   // [2] V stage ready
  B_VT = 10,  // [2] V stage loaded (tail tiles: before the zero fill)
  B_VE = 12,  // [2] V stage free
  B_SF = 14,  // [2] S_x ready
  B_PF = 16,  // [2] P_x written
  B_OF = 18,  // [2] O_x final for the item
  B_OE = 20,  // [2] O_x read by the epilogue
  B_IF = 22,  // [2] item slot published
  B_IE = 24,  // [2] item slot released
  B_XP = 26,  // [4] exchange between the two softmax warps of a row quarter
  B_LF = 30,  // [2] row sums of tile x written for the epilogue, even items
  kNumBars = 32
};
constexpr int kOffItems = kOffBar + kNumBars * 8;  // 2 item slots
constexpr int kOffXch = kOffItems + 2 * 48;        // [4 quarters][2 slots][2 halves][32] floats
constexpr int kOffCtl = kOffXch + 4 * 2 * 2 * 32 * 4;  // TMEM address, abort flag
constexpr int kOffBarLF1 = kOffCtl + 16;           // [2] the same for odd items
constexpr int kSmemBytes = kOffBarLF1 + 16 + 1024;  // + alignment slack

struct Item {
  int r, qt, ha, hb;  // hb < 0: single-tile item
  int g, q0, n, L;
  int ctx, nkv, pad0, pad1;
};

// a prefill entry written by the plan kernel, read through L2
__device__ __forceinline__ PreEntry load_entry(const PreEntry* p) {
  const int4 w0 = __ldcg(reinterpret_cast<const int4*>(p));
  const int4 w1 = __ldcg(reinterpret_cast<const int4*>(p) + 1);
  return PreEntry{w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
}

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
  return (1u << 4)                         // D format f32
         | (1u << 7)                       // A format bf16
         | (1u << 10)                      // B format bf16
         | ((b_mn_major ? 1u : 0u) << 16)  // B major-ness
         | ((128u >> 3) << 17)             // N
         | ((128u >> 4) << 24);            // M
}

// The MMA role runs on a whole converged warp, so that operands are
// warp-uniform values; one elected lane (the lowest, the same every time, so
// that its commits track all its MMAs) issues each instruction.
// D (TMEM) (+)= A (shared) * B (shared)
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D (TMEM) (+)= A (TMEM) * B (shared)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                       uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, e;\n setp.ne.b32 p, %4, 0;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
      " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(
          bar)
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

#define PKV_ST32U(taddr, v)                                                                    \
  asm volatile(                                                                                \
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12," \
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"  \
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),        \
      "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),         \
      "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]),     \
      "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),     \
      "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])                              \
      : "memory")

#define PKV_LD16(taddr, v)                                                                     \
  asm volatile(                                                                                \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
      "%14,%15}, [%16];\n"                                                                     \
      : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]), "=f"(v[6]),   \
        "=f"(v[7]), "=f"(v[8]), "=f"(v[9]), "=f"(v[10]), "=f"(v[11]), "=f"(v[12]),            \
        "=f"(v[13]), "=f"(v[14]), "=f"(v[15])                                                  \
      : "r"(taddr))

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, AttnArgs a, Workspace ws) {
  // This grid is the programmatic dependent of the decode grid, which
  // triggers it after its own wait for the plan kernel: the plan is complete
  // when any CTA here runs, so the items start without waiting for the decode
  // grid (which leaves some SMs to them, see pkv_decode.cu); what the plan and
  // the kernels before it wrote is read through L2 (ld.global.cg).  The split
  // decode results are merged at the end, once the decode grid has finished
  // (so this grid finishing implies that every kernel before it has).
  const int n_pre = __ldcg(&ws.hdr->n_pre_entries);
  if (n_pre == 0) {  // a step without prefill work (every CTA agrees)
    grid_dep_wait();
    combine_splits(a, ws, blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5),
                   gridDim.x * (kThreads / 32));
    return;
  }
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBar;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  // row sums of tile x of item it_cnt written
  auto lf_bar = [&](uint32_t it_cnt, int x) {
    return (it_cnt & 1) ? sbase + kOffBarLF1 + 8u * (uint32_t)x : bar(B_LF + x);
  };
  volatile int* ctl = reinterpret_cast<volatile int*>(smem + kOffCtl);
  volatile int* abort = ctl + 1;  // ctl[0] = TMEM base address
  Item* items = reinterpret_cast<Item*>(smem + kOffItems);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.hq / a.hkv;
  const bool pairs = (G % 2) == 0;  // two heads of one KV head per item
  const int per_entry = pairs ? a.hq / 2 : a.hq;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(B_PF + x), 8);  // one arrival per softmax warp (each writes half of P)
      mbar_init(bar(B_OE + x), 4);  // one arrival per epilogue warp
      mbar_init(bar(B_LF + x), 8);  // one arrival per softmax warp
      mbar_init(sbase + kOffBarLF1 + 8 * x, 8);
      mbar_init(bar(B_IE + x), 1 + 8 + 4);  // MMA warp, softmax warps, epilogue warps
    }
    for (int i = 0; i < 4; ++i) mbar_init(bar(B_XP + i), 2);
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
  const int n_items = n_pre * per_entry;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    // Global loads are issued one step before their values are needed: the
    // next item's cursor and entry (which carries its request's lengths)
    // while the current item is being issued, and each tile's block ids one
    // tile ahead; a load only stalls at its first use.
    uint32_t tile_cnt = 0, vt_uses[kStages] = {0, 0}, qx_cnt[2] = {0, 0};
    int w_nxt = 0;
    if (lane == 0) w_nxt = atomicAdd(&ws.hdr->pre_counter, 1);
    w_nxt = __shfl_sync(0xffffffffu, w_nxt, 0);
    const PreEntry none{-1, 0, 0, 0, 0, 0, 0, 0};
    PreEntry e_nxt = w_nxt < n_items ? load_entry(ws.pre + w_nxt / per_entry) : none;
    for (uint32_t it_cnt = 0;; ++it_cnt) {
      const int slot = it_cnt & 1;
      const int w = w_nxt;
      const PreEntry e = e_nxt;
      const int q0 = e.q0, q1 = e.q0 + e.n, Lr = e.L;
      if (it_cnt >= 2 &&
          !mbar_wait_warp(bar(B_IE + slot), ((it_cnt >> 1) - 1) & 1, abort, ws.err))
        break;
      if (w >= n_items || *abort) {
        if (lane == 0) {
          items[slot].r = -1;
          mbar_arrive(bar(B_IF + slot));
        }
        break;
      }
      Item it;
      {
        const int hp = w % per_entry;
        it.r = e.r;
        it.qt = e.qt;
        it.nkv = e.nkv;
        it.ha = pairs ? 2 * hp : hp;
        it.hb = pairs ? 2 * hp + 1 : -1;
        it.g = it.ha / G;
        it.q0 = q0;
        it.n = q1 - q0;
        it.L = Lr;
        it.ctx = Lr - it.n;
        it.pad0 = it.pad1 = 0;
      }
      if (lane == 0) {
        items[slot] = it;
        mbar_arrive(bar(B_IF + slot));
      }
      // the next item's cursor and entry (consumed after this item)
      if (lane == 0) w_nxt = atomicAdd(&ws.hdr->pre_counter, 1);
      w_nxt = __shfl_sync(0xffffffffu, w_nxt, 0);
      e_nxt = w_nxt < n_items ? load_entry(ws.pre + w_nxt / per_entry) : none;
      const int* btrow = a.bt + (int64_t)it.r * a.bt_width;
      const int row0 = it.q0 + it.qt * kPreTileQ;
      // Q tiles, once the previous item's last S has read them
      bool ok = true;
      for (int x = 0; x < 2 && ok; ++x) {
        const int h = x == 0 ? it.ha : it.hb;
        if (h < 0) continue;
        if (qx_cnt[x] > 0 &&
            !mbar_wait_warp(bar(B_QE + x), (qx_cnt[x] - 1) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        qx_cnt[x]++;
        if (lane == 0) {
          const uint32_t qd = sbase + kOffQ + x * kTileBytes;
          mbar_expect_tx(bar(B_QF + x), kTileBytes);
          tma_load_3d(qd, &tm_q, bar(B_QF + x), 0, h, row0);
          tma_load_3d(qd + kHalfBytes, &tm_q, bar(B_QF + x), 64, h, row0);
        }
      }
      // lane p < pages(j) holds the block id of page p of tile j
      auto tile_pages = [&](int j) { return min(8, (it.L - j * kTileK + 15) / 16); };
      int blk_nxt = lane < tile_pages(0) ? __ldcg(btrow + lane) : 0;
      for (int j = 0; ok && j < it.nkv; ++j) {
        const uint32_t c = tile_cnt++;
        const int s = c % kStages;
        const int key0 = j * kTileK;
        const int pages = tile_pages(j);
        const bool tail = key0 + kTileK > it.L;
        int blk = blk_nxt;
        if (j + 1 < it.nkv && lane < tile_pages(j + 1))
          blk_nxt = __ldcg(btrow + ((key0 + kTileK) >> 4) + lane);
        if (c >= (uint32_t)kStages &&
            !mbar_wait_warp(bar(B_KE + s), ((c / kStages) - 1) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        if (lane < pages && (blk < 0 || (int64_t)blk >= a.num_blocks)) {
          atomicOr(ws.err, PKV_DEV_ERR_BLOCK_ID);
          blk = 0;
        }
        const uint32_t kdst = sbase + kOffK + s * kTileBytes;
        if (lane == 0) mbar_expect_tx(bar(B_KF + s), pages * 2 * kPageBoxBytes);
        __syncwarp();
        if (lane < pages) {
          tma_load_4d(kdst + lane * kPageBoxBytes, &tm_k, bar(B_KF + s), 0, it.g, 0, blk);
          tma_load_4d(kdst + kHalfBytes + lane * kPageBoxBytes, &tm_k, bar(B_KF + s), 64, it.g,
                      0, blk);
        }
        if (c >= (uint32_t)kStages &&
            !mbar_wait_warp(bar(B_VE + s), ((c / kStages) - 1) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        const uint32_t vdst = sbase + kOffV + s * kTileBytes;
        const uint32_t vbar = tail ? bar(B_VT + s) : bar(B_VF + s);
        if (lane == 0) mbar_expect_tx(vbar, pages * 2 * kPageBoxBytes);
        __syncwarp();
        if (lane < pages) {
          tma_load_4d(vdst + lane * kPageBoxBytes, &tm_v, vbar, 0, it.g, 0, blk);
          tma_load_4d(vdst + kHalfBytes + lane * kPageBoxBytes, &tm_v, vbar, 64, it.g, 0, blk);
        }
        if (tail) {
          // wait for the V boxes, zero the rows of keys >= seq_len, publish
          ok = mbar_wait_warp(bar(B_VT + s), vt_uses[s] & 1, abort, ws.err);
          vt_uses[s]++;
          if (!ok) break;
          const int z0 = it.L - key0;
          uint8_t* v = smem + kOffV + s * kTileBytes;
          for (int i = lane; i < (kTileK - z0) * 16; i += 32) {
            const int row = z0 + (i >> 4), within = i & 15;
            *reinterpret_cast<uint4*>(v + (within >> 3) * kHalfBytes + row * 128 +
                                      (within & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_VF + s));
        }
      }
      if (!ok) break;
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    // (the whole warp runs this, in step; see mma_ss)
    {
      const uint32_t id_s = idesc_bf16(false), id_o = idesc_bf16(true);
      uint32_t tile_cnt = 0, s_cnt[2] = {0, 0}, o_cnt[2] = {0, 0}, q_cnt[2] = {0, 0};
      // Operand descriptors of every buffer, built once: a descriptor's low
      // field is the address / 16, so a k-step's offset is added to it.
      const uint64_t dq0 = sdesc(sbase + kOffQ, 16), dq1 = sdesc(sbase + kOffQ + kTileBytes, 16);
      const uint64_t dk0 = sdesc(sbase + kOffK, 16), dk1 = sdesc(sbase + kOffK + kTileBytes, 16);
      const uint64_t dv0 = sdesc(sbase + kOffV, kHalfBytes);
      const uint64_t dv1 = sdesc(sbase + kOffV + kTileBytes, kHalfBytes);
      static_assert(kStages == 2, "one descriptor per stage");
      // S_x(c) = Q_x K_c^T
      auto issue_s = [&](int x, uint32_t c) {
        const uint64_t da = x ? dq1 : dq0, db = (c & 1) ? dk1 : dk0;
        const uint32_t d = tmem + x * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          mma_ss(d, da + off, db + off, id_s, kk > 0);
        }
        mma_commit(bar(B_SF + x));
        s_cnt[x]++;
      };
      // O_x (+)= P_x V_c  (P_x: bf16 pairs, keys 0-63 in columns 0-31 and keys
      // 64-127 in columns 64-95 of S_x: each half where its own scores were)
      auto issue_pv = [&](int x, uint32_t c, bool acc) {
        const uint64_t db = (c & 1) ? dv1 : dv0;
        const uint32_t d = tmem + 256 + x * 128, pa = tmem + x * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(d, pa + (kk >> 2) * 64 + (kk & 3) * 8, db + ((kk * 16 * 128) >> 4), id_o,
                 (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      for (uint32_t it_cnt = 0; ok; ++it_cnt) {
        const int slot = it_cnt & 1;
        if (!mbar_wait_warp(bar(B_IF + slot), (it_cnt >> 1) & 1, abort, ws.err)) break;
        const Item it = items[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_IE + slot));
        if (it.r < 0) break;
        const int nx = it.hb >= 0 ? 2 : 1;
        for (int x = 0; x < nx && ok; ++x)
          ok = mbar_wait_warp(bar(B_QF + x), q_cnt[x]++ & 1, abort, ws.err);
        const uint32_t c0 = tile_cnt;
        if (!ok || !mbar_wait_warp(bar(B_KF + c0 % kStages), (c0 / kStages) & 1, abort, ws.err)) break;
        tc_fence_after();
        for (int x = 0; x < nx; ++x) issue_s(x, c0);
        mma_commit(bar(B_KE + c0 % kStages));
        if (it.nkv == 1)
          for (int x = 0; x < nx; ++x) mma_commit(bar(B_QE + x));
        for (int j = 0; j < it.nkv && ok; ++j) {
          const uint32_t c = c0 + j;
          const bool more = j + 1 < it.nkv;
          if (!mbar_wait_warp(bar(B_VF + c % kStages), (c / kStages) & 1, abort, ws.err)) {
            ok = false;
            break;
          }
          for (int x = 0; x < nx; ++x) {
            if (!mbar_wait_warp(bar(B_PF + x), (s_cnt[x] - 1) & 1, abort, ws.err) ||
                (j == 0 && o_cnt[x] > 0 &&
                 !mbar_wait_warp(bar(B_OE + x), (o_cnt[x] - 1) & 1, abort, ws.err))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(x, c, j > 0);
            if (x == nx - 1) mma_commit(bar(B_VE + c % kStages));  // every PV of V_c issued
            if (more) {
              // the next K tile is waited for only now, with PV_x already queued
              if (x == 0 && !mbar_wait_warp(bar(B_KF + (c + 1) % kStages), ((c + 1) / kStages) & 1,
                                           abort, ws.err)) {
                ok = false;
                break;
              }
              tc_fence_after();
              issue_s(x, c + 1);
            } else {
              mma_commit(bar(B_OF + x));  // O_x final: its epilogue need not wait for the other tile
              o_cnt[x]++;
            }
          }
          if (!ok) break;
          if (more) {
            mma_commit(bar(B_KE + (c + 1) % kStages));
            if (j + 2 == it.nkv)
              for (int x = 0; x < nx; ++x) mma_commit(bar(B_QE + x));
          }
        }
        if (!ok) break;
        tile_cnt += it.nkv;
      }
    }
    __syncwarp();
  } else if (warp < 10) {
    // ------------------- softmax: two warps per row, a column half each -------------------
    // Warp w reads TMEM lanes 32 * (w % 4) .. + 31 (its 32 rows, one per
    // thread) and key columns 64 * hf .. 64 * hf + 63, hf = (w - 2) / 4, of
    // both query tiles of the item in turn; both warps of a row quarter (w and
    // w + 4) sit on the same SM sub-partition and work on the same tile at the
    // same time, so each tile's softmax takes half as long.  The warps of a
    // quarter exchange per-row values (the need for a max pass, the partial
    // maxima, the partial sums) through shared memory and a two-arrival
    // mbarrier, whose waits are bounded like every other.
    const int hf = (warp - 2) >> 2;
    const int qd = warp & 3;
    const int row = qd * 32 + lane;  // == TMEM lane
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    float* xch = reinterpret_cast<float*>(smem + kOffXch);
    const float sl2 = a.scale * kLog2e;
    uint32_t s_cnt[2] = {0, 0}, x_cnt = 0;
    bool ok = true;
    // this lane's value out, the other warp's value for the same row back
    auto exchange = [&](float v) -> float {
      const int sl = x_cnt & 1;  // two slots: a slot is rewritten only after both read it
      xch[((qd * 2 + sl) * 2 + hf) * 32 + lane] = v;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_XP + qd));
      if (!mbar_wait_warp(bar(B_XP + qd), x_cnt & 1, abort, ws.err)) ok = false;
      x_cnt++;
      return xch[((qd * 2 + sl) * 2 + (1 - hf)) * 32 + lane];
    };
    float* lsum = reinterpret_cast<float*>(smem + kOffLsum);
    for (uint32_t it_cnt = 0; ok; ++it_cnt) {
      const int slot = it_cnt & 1;
      if (!mbar_wait_warp(bar(B_IF + slot), (it_cnt >> 1) & 1, abort, ws.err)) break;
      const Item it = items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_IE + slot));
      if (it.r < 0) break;
      const int nx = it.hb >= 0 ? 2 : 1;
      const int qrow = it.qt * kPreTileQ + row;  // row inside the request
      const bool valid_row = qrow < it.n;
      const int qpos = valid_row ? it.ctx + qrow : 0;  // last visible key
      float m_used[2] = {-INFINITY, -INFINITY}, l_part[2] = {0.f, 0.f};
      for (int j = 0; j < it.nkv && ok; ++j) {
        const int lim = qpos - j * kTileK - 64 * hf;  // my columns <= lim are visible
        const bool masked = !__all_sync(0xffffffffu, lim >= 63);
        for (int x = 0; x < nx && ok; ++x) {
          if (!mbar_wait_warp(bar(B_SF + x), s_cnt[x]++ & 1, abort, ws.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t t_s = tmem + x * 128 + 64 * hf + lane_off;
          // my 64 scores of the row in registers (one wait), then P in place
          float sv[64];
          auto load_scores = [&]() {
            PKV_LD32(t_s + 0, (sv + 0));
            PKV_LD32(t_s + 32, (sv + 32));
            tmem_wait_ld();
            if (masked) {
#pragma unroll
              for (int i = 0; i < 64; ++i) sv[i] = (i <= lim) ? sv[i] : -INFINITY;
            }
          };
          // p = exp2(s * scale * log2(e) - m) two columns at a time (packed
          // fp32 pairs for the multiply-add and the sums); the bf16 pairs are
          // packed over sv[0..31] (sv[2i], sv[2i+1] read before sv[i] is written)
          float rs[4];
          auto exp_pack = [&](float m) {
            rs[0] = rs[1] = rs[2] = rs[3] = 0.f;
            const float nm = -m;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              float x0, x1;
              fma2(x0, x1, sv[2 * i], sv[2 * i + 1], sl2, sl2, nm, nm);
              const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
              add2(rs[2 * (i & 1)], rs[2 * (i & 1) + 1], p0, p1);
              sv[i] = __uint_as_float(pack_bf16(p0, p1));
            }
          };
          load_scores();
          float alpha = 1.f;
          bool resc = false;
          // After the first tile, P is computed with the running max straight
          // away: no p exceeds 2^8 (the rescale threshold) while a half-row
          // sum does not, so the max pass is taken only when some half-row's
          // sum does (or is not finite) in either warp of the quarter.
          bool need_max = j == 0;
          if (!need_max) {
            exp_pack(m_used[x]);
            const float tot = (rs[0] + rs[1]) + (rs[2] + rs[3]);
            const float mine = (tot <= 256.f) ? 0.f : 1.f;
            const float other = exchange(mine);
            if (!ok) break;
            need_max = __any_sync(0xffffffffu, mine + other > 0.f);
            if (need_max) load_scores();
          }
          if (need_max) {
            // the row maximum over both halves: three-input max chains, then
            // the other warp's half through the exchange
            float mx[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) mx[k] = max3f(sv[k], sv[k + 4], sv[k + 8]);
#pragma unroll
            for (int i = 12; i < 60; i += 8)
#pragma unroll
              for (int k = 0; k < 4; ++k) mx[k] = max3f(mx[k], sv[i + k], sv[i + 4 + k]);
#pragma unroll
            for (int k = 0; k < 4; ++k) mx[k] = fmaxf(mx[k], sv[60 + k]);
            const float pm = fmaxf(max3f(mx[0], mx[1], mx[2]), mx[3]);
            const float po = exchange(pm);
            if (!ok) break;
            // (both warps form the same value: the halves in a fixed order)
            const float mt = (hf == 0 ? fmaxf(pm, po) : fmaxf(po, pm)) * sl2;
            resc = mt > m_used[x] + kRescaleThreshold;
            if (resc) {
              alpha = fast_exp2(m_used[x] - mt);  // 0 on the first tile
              m_used[x] = mt;
            }
            exp_pack(m_used[x]);
          }
          PKV_ST32(t_s, (sv + 0));  // P half: 32 packed columns where my scores began
          l_part[x] = l_part[x] * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
          if (j > 0 && __any_sync(0xffffffffu, resc)) {
            // PV(j-1) is complete (S(j) is, and one thread's MMAs finish in
            // order); each warp rescales its own 64 output columns
            const uint32_t t_o = tmem + 256 + x * 128 + 64 * hf + lane_off;
#pragma unroll
            for (int ch = 0; ch < 2; ++ch) {
              float ov[32];
              PKV_LD32(t_o + ch * 32, ov);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] *= alpha;
              PKV_ST32(t_o + ch * 32, ov);
            }
          }
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_PF + x));
        }
      }
      if (!ok) break;
      // this warp's partial row sums of the item, for the epilogue warps
      // (one barrier per item parity: the softmax may finish the next item
      // before the epilogue has waited for this one, and one barrier would
      // then have completed two phases, which a parity wait cannot tell
      // apart from none)
      for (int x = 0; x < nx; ++x) {
        lsum[(((it_cnt & 1) * 2 + x) * 2 + hf) * 128 + row] = l_part[x];
        __syncwarp();
        if (lane == 0) mbar_arrive(lf_bar(it_cnt, x));
      }
    }
  } else {
    // ------------------ epilogue: one warp per TMEM lane quarter ------------------
    // Warp w (10..13) owns rows 32 * (w % 4) .. + 31 of both output tiles.  When
    // O_x is final (its last P.V done) and both partial row sums are in, the
    // warp reads the 128-column row block out of TMEM in two halves,
    // normalises them and packs them to bf16 in registers, and releases O_x as
    // soon as the second half is read (the next item's first P.V may then
    // overwrite it); each 32-column chunk goes out through the warp's staging
    // area in shared memory, so that each global store writes whole 64-byte
    // row pieces (8 rows x 4 lanes).
    // The softmax warps never wait for this work.
    const int qd = warp & 3;
    const int row = qd * 32 + lane;  // == TMEM lane
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const float* lsum = reinterpret_cast<const float*>(smem + kOffLsum);
    const uint32_t stg = sbase + kOffStage + (warp - 10) * kStageWarp;
    uint32_t o_cnt[2] = {0, 0};
    for (uint32_t it_cnt = 0;; ++it_cnt) {
      const int slot = it_cnt & 1;
      if (!mbar_wait_warp(bar(B_IF + slot), (it_cnt >> 1) & 1, abort, ws.err)) break;
      const Item it = items[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_IE + slot));
      if (it.r < 0) break;
      const int nx = it.hb >= 0 ? 2 : 1;
      bool ok = true;
      for (int x = 0; x < nx && ok; ++x) {
        const uint32_t par = o_cnt[x]++ & 1;
        if (!mbar_wait_warp(bar(B_OF + x), par, abort, ws.err) ||
            !mbar_wait_warp(lf_bar(it_cnt, x), (it_cnt >> 1) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float* ls = lsum + ((it_cnt & 1) * 2 + x) * 2 * 128;
        const float inv = 1.f / (ls[row] + ls[128 + row]);  // the two column halves' sums
        const uint32_t t_o = tmem + 256 + x * 128 + lane_off;
        const int h = x == 0 ? it.ha : it.hb;
        const int row_base = it.qt * kPreTileQ + qd * 32;  // the warp's first row
        uint16_t* obase = a.out + (int64_t)it.q0 * a.out_stride + (int64_t)h * kHeadSize;
        // two 64-column halves; O_x is released once the second half is in
        // registers (the first half is already on its way out by then)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t held[32];  // 64 outputs of the row, bf16 pairs
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            float ov[16];
            PKV_LD16(t_o + half * 64 + ch * 16, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i)
              held[ch * 8 + i] = pack_bf16(ov[2 * i] * inv, ov[2 * i + 1] * inv);
          }
          if (half == 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_OE + x));
          }
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            // this lane's row: 16-byte piece k at slot k ^ ((lane >> 1) & 3), so
            // that eight lanes of a store phase hit eight different bank groups
#pragma unroll
            for (int k = 0; k < 4; ++k)
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};\n" ::"r"(
                               stg + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4)),
                           "r"(held[cc * 16 + 4 * k]), "r"(held[cc * 16 + 4 * k + 1]),
                           "r"(held[cc * 16 + 4 * k + 2]), "r"(held[cc * 16 + 4 * k + 3])
                           : "memory");
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int rr = i * 8 + (lane >> 2), c = lane & 3;
              uint4 v;
              asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];\n"
                           : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                           : "r"(stg + rr * 64 + ((c ^ ((rr >> 1) & 3)) << 4))
                           : "memory");
              const int qr = row_base + rr;
              if (qr < it.n)
                *reinterpret_cast<uint4*>(obase + (int64_t)qr * a.out_stride + half * 64 +
                                          cc * 32 + c * 8) = v;
            }
            __syncwarp();
          }
        }
      }
      if (!ok) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem),
                 "r"(kTmemCols));
  }
  // the split decode results, once the decode grid has finished
  grid_dep_wait();
  combine_splits(a, ws, blockIdx.x * (kThreads / 32) + warp, gridDim.x * (kThreads / 32));
}

}  // namespace

cudaError_t launch_prefill(const AttnArgs& a, const Workspace& ws, int sms, cudaStream_t st) {
  static std::atomic<bool> attr[kMaxAttrDevices];
  if (cudaError_t e = smem_attr_once(prefill_kernel, kSmemBytes, attr)) return e;
  CUtensorMap tq, tk, tv;
  if (!make_rows_map(&tq, a.q, a.q_rows, a.hq, a.q_stride, 1, kPreTileQ) ||
      !make_cache_map(&tk, a.kc, a.num_blocks, a.hkv) ||
      !make_cache_map(&tv, a.vc, a.num_blocks, a.hkv))
    return cudaErrorInvalidValue;
  return launch_dependent(prefill_kernel, dim3(sms), dim3(kThreads), kSmemBytes, st, tq, tk, tv,
                          a, ws);
}

}  // namespace pkv
