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
// and "b" share every K/V tile.  Keys are taken 64 at a time.  Tensor memory
// (512 columns) holds each query tile's output O (128 columns) and two score
// buffers S[0], S[1] (64 columns each): while the softmax works on the scores
// of key tile j, the tensor cores already hold those of tile j + 1 and compute
// P.V of tile j - 1 and S of tile j + 1's successor, so a query tile's chain
// (scores -> softmax -> P.V) never waits for its own next scores.  A
// persistent grid (one CTA per SM) takes items from an atomic cursor, longest
// first, and treats the key tiles of consecutive items as one stream.  Roles:
//   warp 0      K producer: publishes items in a four-slot ring, loads the
//               two Q tiles of an item by TMA into one of two Q buffers, and
//               the K tiles (4 pages, one 16-slot x 64-dim box per page and
//               half, 128-byte swizzle) into a 3-stage ring;
//   warp 14     V producer: the V tiles into a 2-stage ring; in a request's
//               last tile it zero-fills the V rows of keys past seq_len so
//               that no stale value (NaN) reaches P.V;
//   warp 1      allocates TMEM and issues every MMA from one thread: S_x(g) =
//               Q_x K_g^T into S_x[g % 2] as soon as P.V of tile g - 2 (which
//               read that buffer) is issued, and O_x += P_x(g) V_g with P
//               taken from TMEM (the scores' first 32 columns, overwritten
//               with bf16 probabilities) and V from shared memory (MN-major);
//               tcgen05.commit drives the mbarriers;
//   warps 2-9   softmax, one warp per (query tile, TMEM lane quarter), one
//               query row per thread: scores -> causal/length mask (only on
//               tiles that cross the diagonal) -> running max in the log2
//               domain -> exp2 -> row sum -> bf16 P back into TMEM.  O is
//               rescaled in TMEM only when a row's max grows by more than 2^8
//               (exact, rare), after P.V of the previous tile is complete;
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

constexpr int kThreads = 480;                     // 15 warps
constexpr int kTileK = 64;                        // keys per KV tile
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kItemSlots = 4;
constexpr int kQHalf = 128 * 128;                 // 128 query rows x 64 bf16
constexpr int kQTile = 2 * kQHalf;                // 32 KB
constexpr int kKVHalf = kTileK * 128;             // 64 keys x 64 bf16
constexpr int kKVTile = 2 * kKVHalf;              // 16 KB
constexpr int kPageBoxBytes = 16 * 128;           // one 16-slot x 64-dim box
constexpr int kTmemCols = 512;
constexpr int kColS = 256;                        // S_x[p] at kColS + 128 x + 64 p; O_x at 128 x
constexpr float kRescaleThreshold = 8.0f;         // log2 units

// shared-memory layout (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;                          // Q(x, buffer b) at kOffQ + (2 x + b) kQTile
constexpr int kOffK = kOffQ + 4 * kQTile;
constexpr int kOffV = kOffK + kKStages * kKVTile;
constexpr int kStageWarp = 32 * 64;               // epilogue staging: 32 rows x 64 bytes
constexpr int kOffStage = kOffV + kVStages * kKVTile;  // one staging area per epilogue warp
constexpr int kOffLsum = kOffStage + 4 * kStageWarp;   // [item slot][tile][128 rows] floats
constexpr int kOffBar = kOffLsum + kItemSlots * 2 * 128 * 4;
enum {
  B_QF = 0,   // [2 x + b] Q tile loaded
  B_QE = 4,   // [2 x + b] Q buffer read by the item's last S
  B_KF = 8,   // [3] K stage loaded
  B_KE = 11,  // [3] K stage free
  B_VF = 14,  // [2] V stage ready
  B_VT = 16,  // [2] V stage loaded (tail tiles: before the zero fill)
  B_VE = 18,  // [2] V stage free
  B_SF = 20,  // [2 x + p] S_x[p] ready
  B_PF = 24,  // [2 x + p] P_x written into S_x[p]
  B_PD = 28,  // [x] a P.V into O_x complete
  B_OF = 30,  // [x] O_x final for the item
  B_OE = 32,  // [x] O_x read by the epilogue
  B_IF = 34,  // [slot] item published
  B_IE = 38,  // [slot] item released by every role
  B_LF = 42,  // [4 x + slot] row sums of tile x written for the epilogue
  kNumBars = 50
};
constexpr int kOffItems = kOffBar + kNumBars * 8;           // kItemSlots items
constexpr int kOffCtl = kOffItems + kItemSlots * 48;        // TMEM address, abort flag
constexpr int kSmemBytes = kOffCtl + 16 + 1024;             // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

struct Item {
  int r, qt, ha, hb;  // hb < 0: single-tile item
  int g, q0, n, L;
  int ctx, nkv, pad0, pad1;  // nkv: 64-key tiles the item reads
};

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

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t n, bool b_mn_major) {
  return (1u << 4)                         // D format f32
         | (1u << 7)                       // A format bf16
         | (1u << 10)                      // B format bf16
         | ((b_mn_major ? 1u : 0u) << 16)  // B major-ness
         | ((n >> 3) << 17)                // N
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
  // This launch also merges the split-KV decode results of the step (the
  // decode kernel ran before it in stream order), which saves a launch of its
  // own: every warp of the grid does it when the batch has no prefill work,
  // else the epilogue warps, before their first output tile is due.
  grid_dep_wait();  // the work lists and the decode kernel's partial results
  if (ws.hdr->n_pre_entries == 0) {  // (every CTA agrees)
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
  volatile int* ctl = reinterpret_cast<volatile int*>(smem + kOffCtl);
  volatile int* abort = ctl + 1;  // ctl[0] = TMEM base address
  Item* items = reinterpret_cast<Item*>(smem + kOffItems);
  float* lsum = reinterpret_cast<float*>(smem + kOffLsum);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.hq / a.hkv;
  const bool pairs = (G % 2) == 0;  // two heads of one KV head per item
  const int nx = pairs ? 2 : 1;
  const int per_entry = pairs ? a.hq / 2 : a.hq;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
    for (int i = 0; i < 4; ++i) mbar_init(bar(B_PF + i), 4);  // the four softmax warps of a tile
    for (int x = 0; x < 2; ++x) mbar_init(bar(B_OE + x), 4);  // the four epilogue warps
    for (int i = 0; i < 8; ++i) mbar_init(bar(B_LF + i), 4);  // the four softmax warps of a tile
    // MMA warp, 8 softmax warps, 4 epilogue warps, V producer
    for (int i = 0; i < kItemSlots; ++i) mbar_init(bar(B_IE + i), 1 + 8 + 4 + 1);
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
  const int n_items = ws.hdr->n_pre_entries * per_entry;

  // the item in ring slot n & 3, once published (every role reads it this way)
  auto take_item = [&](uint32_t n, Item* it) -> bool {
    if (!mbar_wait_warp(bar(B_IF + (n & 3)), (n >> 2) & 1, abort, ws.err)) return false;
    *it = items[n & 3];
    __syncwarp();
    return true;
  };
  // pages of key tile j of an item, and whether it holds keys past seq_len
  auto tile_pages = [&](const Item& it, int j) { return min(4, (it.L - j * kTileK + 15) / 16); };

  if (warp == 0) {
    // ------------------------------ K producer ------------------------------
    // Global loads are issued one step before their values are needed: the
    // next item's cursor and entry (which carries its request's lengths)
    // while the current item is being loaded, and each tile's block ids one
    // tile ahead; a load only stalls at its first use.
    uint32_t g = 0;  // K tiles loaded (all items)
    int w_nxt = 0;
    if (lane == 0) w_nxt = atomicAdd(&ws.hdr->pre_counter, 1);
    w_nxt = __shfl_sync(0xffffffffu, w_nxt, 0);
    const PreEntry none{-1, 0, 0, 0, 0, 0, 0, 0};
    PreEntry e_nxt = w_nxt < n_items ? ws.pre[w_nxt / per_entry] : none;
    for (uint32_t it_cnt = 0;; ++it_cnt) {
      const int slot = it_cnt & 3;
      const int w = w_nxt;
      const PreEntry e = e_nxt;
      if (it_cnt >= kItemSlots &&
          !mbar_wait_warp(bar(B_IE + slot), ((it_cnt >> 2) - 1) & 1, abort, ws.err))
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
        it.ha = pairs ? 2 * hp : hp;
        it.hb = pairs ? 2 * hp + 1 : -1;
        it.g = it.ha / G;
        it.q0 = e.q0;
        it.n = e.n;
        it.L = e.L;
        it.ctx = e.L - e.n;
        const int last_row = min(kPreTileQ * (e.qt + 1), e.n);
        it.nkv = (it.ctx + last_row + kTileK - 1) / kTileK;
        it.pad0 = it.pad1 = 0;
      }
      if (lane == 0) {
        items[slot] = it;
        mbar_arrive(bar(B_IF + slot));
      }
      // the next item's cursor and entry (consumed after this item)
      if (lane == 0) w_nxt = atomicAdd(&ws.hdr->pre_counter, 1);
      w_nxt = __shfl_sync(0xffffffffu, w_nxt, 0);
      e_nxt = w_nxt < n_items ? ws.pre[w_nxt / per_entry] : none;
      const int* btrow = a.bt + (int64_t)it.r * a.bt_width;
      const int row0 = it.q0 + it.qt * kPreTileQ;
      // Q tiles into buffer it_cnt & 1, once the item before last has read it
      const int qb = it_cnt & 1;
      bool ok = true;
      for (int x = 0; x < nx && ok; ++x) {
        const int h = x == 0 ? it.ha : it.hb;
        if (it_cnt >= 2 &&
            !mbar_wait_warp(bar(B_QE + 2 * x + qb), ((it_cnt >> 1) - 1) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t qd = sbase + kOffQ + (2 * x + qb) * kQTile;
          mbar_expect_tx(bar(B_QF + 2 * x + qb), kQTile);
          tma_load_3d(qd, &tm_q, bar(B_QF + 2 * x + qb), 0, h, row0);
          tma_load_3d(qd + kQHalf, &tm_q, bar(B_QF + 2 * x + qb), 64, h, row0);
        }
      }
      // lane p < pages(j) holds the block id of page p of tile j
      int blk_nxt = lane < tile_pages(it, 0) ? __ldg(btrow + lane) : 0;
      for (int j = 0; ok && j < it.nkv; ++j) {
        const uint32_t c = g++;
        const int s = c % kKStages;
        const int pages = tile_pages(it, j);
        int blk = blk_nxt;
        if (j + 1 < it.nkv && lane < tile_pages(it, j + 1))
          blk_nxt = __ldg(btrow + (((j + 1) * kTileK) >> 4) + lane);
        if (c >= (uint32_t)kKStages &&
            !mbar_wait_warp(bar(B_KE + s), ((c / kKStages) - 1) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        if (lane < pages && (blk < 0 || (int64_t)blk >= a.num_blocks)) {
          atomicOr(ws.err, PKV_DEV_ERR_BLOCK_ID);
          blk = 0;
        }
        const uint32_t kdst = sbase + kOffK + s * kKVTile;
        if (lane == 0) mbar_expect_tx(bar(B_KF + s), pages * 2 * kPageBoxBytes);
        __syncwarp();
        if (lane < pages) {
          tma_load_4d(kdst + lane * kPageBoxBytes, &tm_k, bar(B_KF + s), 0, it.g, 0, blk);
          tma_load_4d(kdst + kKVHalf + lane * kPageBoxBytes, &tm_k, bar(B_KF + s), 64, it.g, 0,
                      blk);
        }
      }
      if (!ok) break;
    }
  } else if (warp == 14) {
    // ------------------------------ V producer ------------------------------
    uint32_t g = 0, vt_uses[kVStages] = {0, 0};
    for (uint32_t it_cnt = 0;; ++it_cnt) {
      Item it;
      if (!take_item(it_cnt, &it) || it.r < 0) break;
      const int* btrow = a.bt + (int64_t)it.r * a.bt_width;
      bool ok = true;
      int blk_nxt = lane < tile_pages(it, 0) ? __ldg(btrow + lane) : 0;
      for (int j = 0; j < it.nkv; ++j) {
        const uint32_t c = g++;
        const int s = c % kVStages;
        const int key0 = j * kTileK;
        const int pages = tile_pages(it, j);
        const bool tail = key0 + kTileK > it.L;
        int blk = blk_nxt;
        if (j + 1 < it.nkv && lane < tile_pages(it, j + 1))
          blk_nxt = __ldg(btrow + ((key0 + kTileK) >> 4) + lane);
        if (c >= (uint32_t)kVStages &&
            !mbar_wait_warp(bar(B_VE + s), ((c / kVStages) - 1) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        if (lane < pages && (blk < 0 || (int64_t)blk >= a.num_blocks)) blk = 0;  // (K reports it)
        const uint32_t vdst = sbase + kOffV + s * kKVTile;
        const uint32_t vbar = tail ? bar(B_VT + s) : bar(B_VF + s);
        if (lane == 0) mbar_expect_tx(vbar, pages * 2 * kPageBoxBytes);
        __syncwarp();
        if (lane < pages) {
          tma_load_4d(vdst + lane * kPageBoxBytes, &tm_v, vbar, 0, it.g, 0, blk);
          tma_load_4d(vdst + kKVHalf + lane * kPageBoxBytes, &tm_v, vbar, 64, it.g, 0, blk);
        }
        if (tail) {
          // wait for the V boxes, zero the rows of keys >= seq_len, publish
          ok = mbar_wait_warp(bar(B_VT + s), vt_uses[s] & 1, abort, ws.err);
          vt_uses[s]++;
          if (!ok) break;
          const int z0 = it.L - key0;
          uint8_t* v = smem + kOffV + s * kKVTile;
          for (int i = lane; i < (kTileK - z0) * 16; i += 32) {
            const int row = z0 + (i >> 4), within = i & 15;
            *reinterpret_cast<uint4*>(v + (within >> 3) * kKVHalf + row * 128 +
                                      (within & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_VF + s));
        }
      }
      if (!ok) break;
      if (lane == 0) mbar_arrive(bar(B_IE + (it_cnt & 3)));
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    // (the whole warp runs this, in step; see mma_ss)  Two cursors over the
    // stream of key tiles g of consecutive items: P.V of tile g_p, and S of
    // tile g_s <= g_p + 1 (S of tile g overwrites the buffer P.V of tile
    // g - 2 read, so it is issued after that P.V; one thread's MMAs run in
    // order).
    const uint32_t id_s = idesc_bf16(kTileK, false), id_o = idesc_bf16(128, true);
    // Operand descriptors of the first buffer of each kind, built once: a
    // descriptor's low field is the address / 16, so other buffers and
    // k-steps add their offset / 16.
    const uint64_t dq = sdesc(sbase + kOffQ, 16);
    const uint64_t dk = sdesc(sbase + kOffK, 16);
    const uint64_t dv = sdesc(sbase + kOffV, kKVHalf);
    // S_x(g) = Q_x K_g^T into S_x[g % 2]
    auto issue_s = [&](int x, int qb, uint32_t g) {
      const uint64_t da = dq + (((2 * x + qb) * kQTile) >> 4);
      const uint64_t db = dk + (((g % kKStages) * kKVTile) >> 4);
      const uint32_t d = tmem + kColS + x * 128 + (g & 1) * 64;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(d, da + (((kk >> 2) * kQHalf + (kk & 3) * 32) >> 4),
               db + (((kk >> 2) * kKVHalf + (kk & 3) * 32) >> 4), id_s, kk > 0);
      mma_commit(bar(B_SF + 2 * x + (g & 1)));
    };
    // O_x (+)= P_x(g) V_g  (P_x(g): bf16 pairs in the first 32 columns of S_x[g % 2])
    auto issue_pv = [&](int x, uint32_t g, bool acc) {
      const uint64_t db = dv + (((g % kVStages) * kKVTile) >> 4);
      const uint32_t d = tmem + x * 128, pa = tmem + kColS + x * 128 + (g & 1) * 64;
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ts(d, pa + kk * 8, db + ((kk * 16 * 128) >> 4), id_o, (acc || kk > 0) ? 1u : 0u);
      mma_commit(bar(B_PD + x));
    };
    uint32_t n_s = 0, n_p = 0, g_s = 0, g_p = 0, o_cnt[2] = {0, 0};
    int j_s = 0, j_p = 0;
    Item it_s, it_p;
    bool ok = take_item(0, &it_s);
    it_p = it_s;
    bool s_live = ok && it_s.r >= 0;
    while (ok && it_p.r >= 0) {
      // S of the tiles up to one past P.V's, into the next items if need be
      while (s_live && g_s < g_p + 2) {
        if (j_s == it_s.nkv) {
          ++n_s;
          j_s = 0;
          if (!(ok = take_item(n_s, &it_s))) break;
          if (it_s.r < 0) {
            s_live = false;
            break;
          }
        }
        if (j_s == 0)
          for (int x = 0; x < nx && ok; ++x)
            ok = mbar_wait_warp(bar(B_QF + 2 * x + (n_s & 1)), (n_s >> 1) & 1, abort, ws.err);
        if (!ok || !mbar_wait_warp(bar(B_KF + g_s % kKStages), (g_s / kKStages) & 1, abort,
                                   ws.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int x = 0; x < nx; ++x) issue_s(x, n_s & 1, g_s);
        mma_commit(bar(B_KE + g_s % kKStages));
        if (j_s == it_s.nkv - 1)
          for (int x = 0; x < nx; ++x) mma_commit(bar(B_QE + 2 * x + (n_s & 1)));
        ++j_s;
        ++g_s;
      }
      if (!ok) break;
      // P.V of tile g_p
      if (!mbar_wait_warp(bar(B_VF + g_p % kVStages), (g_p / kVStages) & 1, abort, ws.err)) break;
      const bool last = j_p == it_p.nkv - 1;
      for (int x = 0; x < nx && ok; ++x) {
        if (!mbar_wait_warp(bar(B_PF + 2 * x + (g_p & 1)), (g_p >> 1) & 1, abort, ws.err) ||
            (j_p == 0 && o_cnt[x] > 0 &&
             !mbar_wait_warp(bar(B_OE + x), (o_cnt[x] - 1) & 1, abort, ws.err))) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(x, g_p, j_p > 0);
        if (last) {
          mma_commit(bar(B_OF + x));  // O_x final: its epilogue need not wait for the other tile
          o_cnt[x]++;
        }
      }
      if (!ok) break;
      mma_commit(bar(B_VE + g_p % kVStages));  // every P.V of V_g issued
      ++g_p;
      if (++j_p == it_p.nkv) {
        if (lane == 0) mbar_arrive(bar(B_IE + (n_p & 3)));
        ++n_p;
        j_p = 0;
        if (!(ok = take_item(n_p, &it_p))) break;
      }
    }
    __syncwarp();
  } else if (warp < 10) {
    // --------------- softmax: one warp per (query tile, row quarter) ---------------
    // Warp w handles query tile x = (w - 2) / 4 and reads TMEM lanes 32 * (w %
    // 4) .. + 31 (its 32 rows, one per thread), all 64 columns of each score
    // tile; the two warps of an SM sub-partition work on the two query tiles.
    const int x = (warp - 2) >> 2;
    const int qd = warp & 3;
    const int row = qd * 32 + lane;  // == TMEM lane
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const float sl2 = a.scale * kLog2e;
    uint32_t g = 0;  // key tiles of this query tile so far (all items)
    bool ok = true;
    for (uint32_t it_cnt = 0; ok; ++it_cnt) {
      Item it;
      if (!take_item(it_cnt, &it) || it.r < 0) break;
      const int slot = it_cnt & 3;
      if (x >= nx) {  // single-head items: the second tile's warps have no work
        if (lane == 0) mbar_arrive(bar(B_IE + slot));
        continue;
      }
      const int qrow = it.qt * kPreTileQ + row;  // row inside the request
      const bool valid_row = qrow < it.n;
      const int qpos = valid_row ? it.ctx + qrow : 0;  // last visible key
      float m_used = -INFINITY, l_run = 0.f;
      for (int j = 0; j < it.nkv; ++j) {
        const uint32_t c = g++;
        const int p = c & 1;
        const int lim = qpos - j * kTileK;  // columns <= lim are visible
        const bool masked = !__all_sync(0xffffffffu, lim >= kTileK - 1);
        if (!mbar_wait_warp(bar(B_SF + 2 * x + p), (c >> 1) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t_s = tmem + kColS + x * 128 + p * 64 + lane_off;
        // the row's 64 scores in registers (one wait), then P in place
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
        // After an item's first tile, P is computed with the running max
        // straight away: no p exceeds 2^8 (the rescale threshold) while the
        // row sum does not, so the max pass is taken only when some row's sum
        // in the warp does (or is not finite).
        bool need_max = j == 0;
        if (!need_max) {
          exp_pack(m_used);
          const float tot = (rs[0] + rs[1]) + (rs[2] + rs[3]);
          need_max = __any_sync(0xffffffffu, !(tot <= 256.f));
          if (need_max) load_scores();
        }
        if (need_max) {
          // the row maximum: three-input max chains
          float mx[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) mx[k] = max3f(sv[k], sv[k + 4], sv[k + 8]);
#pragma unroll
          for (int i = 12; i < 60; i += 8)
#pragma unroll
            for (int k = 0; k < 4; ++k) mx[k] = max3f(mx[k], sv[i + k], sv[i + 4 + k]);
#pragma unroll
          for (int k = 0; k < 4; ++k) mx[k] = fmaxf(mx[k], sv[60 + k]);
          const float mt = fmaxf(max3f(mx[0], mx[1], mx[2]), mx[3]) * sl2;
          resc = mt > m_used + kRescaleThreshold;
          if (resc) {
            alpha = fast_exp2(m_used - mt);  // 0 on the first tile
            m_used = mt;
          }
          exp_pack(m_used);
        }
        PKV_ST32(t_s, (sv + 0));  // P: 32 packed columns where the scores began
        l_run = l_run * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
          // O_x holds P.V of the item's tiles up to j - 1 once that P.V is
          // complete; rescale the warp's 32 rows (128 columns)
          if (!mbar_wait_warp(bar(B_PD + x), (c - 1) & 1, abort, ws.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t t_o = tmem + x * 128 + lane_off;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
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
        if (lane == 0) mbar_arrive(bar(B_PF + 2 * x + p));
      }
      if (!ok) break;
      // the row sums of the item, for the epilogue warps
      lsum[(slot * 2 + x) * 128 + row] = l_run;
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_LF + 4 * x + slot));
        mbar_arrive(bar(B_IE + slot));
      }
    }
  } else {
    // ------------------ epilogue: one warp per TMEM lane quarter ------------------
    // Warp w (10..13) owns rows 32 * (w % 4) .. + 31 of both output tiles.  When
    // O_x is final (its last P.V done) and the row sums are in, the warp reads
    // the 128-column row block out of TMEM in two halves, normalises them and
    // packs them to bf16 in registers, and releases O_x as soon as the second
    // half is read (the next item's first P.V may then overwrite it); each
    // 32-column chunk goes out through the warp's staging area in shared
    // memory, so that each global store writes whole 64-byte row pieces (8
    // rows x 4 lanes).  The softmax warps never wait for this work.
    const int qd = warp & 3;
    const int row = qd * 32 + lane;  // == TMEM lane
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    const uint32_t stg = sbase + kOffStage + (warp - 10) * kStageWarp;
    combine_splits(a, ws, blockIdx.x * 4 + (warp - 10), gridDim.x * 4);
    uint32_t o_cnt[2] = {0, 0};
    for (uint32_t it_cnt = 0;; ++it_cnt) {
      Item it;
      if (!take_item(it_cnt, &it) || it.r < 0) break;
      const int slot = it_cnt & 3;
      bool ok = true;
      for (int x = 0; x < nx && ok; ++x) {
        if (!mbar_wait_warp(bar(B_OF + x), o_cnt[x]++ & 1, abort, ws.err) ||
            !mbar_wait_warp(bar(B_LF + 4 * x + slot), (it_cnt >> 2) & 1, abort, ws.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float inv = 1.f / lsum[(slot * 2 + x) * 128 + row];
        const uint32_t t_o = tmem + x * 128 + lane_off;
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
      if (lane == 0) mbar_arrive(bar(B_IE + slot));
    }
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
