// Step plan: turns the device-resident batch metadata into work lists.
//
// "Tour: One forward pass", stop 5: the attention metadata carries
// query_start_loc, seq_lens and the block table; its max_query_len /
// max_seq_len come from CPU mirrors.  Here the host never reads the device
// metadata (no device-to-host copy, so a step can be captured in a CUDA
// graph): one small kernel reads query_start_loc and seq_lens on the device,
// checks them, and writes
//   * decode units (request, KV head, key range) for requests whose query
//     tokens x heads of a KV head fit one decode unit's rows (single-token
//     and short multi-token steps), split along the keys so that the
//     persistent decode grid has several units per worker (split-KV);
//   * split pairs: the (request, KV head) pairs whose splits are merged
//     afterwards (pkv_combine.cuh);
//   * prefill entries (request, 128-row query tile) for longer requests,
//     ordered longest first;
//   * a header with the counts, the split size and zeroed scheduler cursors.
// The kernel runs a few CTAs: each one reads the whole metadata and forms
// every offset (the scans are cheap and the same in every CTA), then writes
// its share of the entries — one request per warp of the grid — so that a
// batch of hundreds of requests and tens of thousands of units is not
// written by a single SM.  A CTA has as many threads as the batch has
// requests (rounded up to a warp, at most 1024): the plan's cost is a chain
// of block-wide barriers and scans, so a small batch plans with one warp.
// "vLLM MHA Code Path: From QKV to Paged KV Cache", section "Prefill and
// decode share an interface": the phase of a request is told apart only by
// its query and sequence lengths, which is what this kernel does.
#include <algorithm>
#include <climits>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kPlanThreads = 1024;  // the most threads of a plan CTA

// Exclusive block-wide prefix sums of eight ints per thread (two int4; any
// whole number of warps up to 32), the eight scans sharing their barriers;
// *tx / *ty receive the block totals.
__device__ void block_exclusive_scan8(int4 x, int4 y, int4* ox, int4* oy, int4* tx, int4* ty,
                                      int4* sx, int4* sy) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  auto add4 = [](int4 a, int4 b) { return make_int4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w); };
  auto sub4 = [](int4 a, int4 b) { return make_int4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w); };
  auto shfl_up4 = [](int4 v, int o) {
    return make_int4(__shfl_up_sync(0xffffffffu, v.x, o), __shfl_up_sync(0xffffffffu, v.y, o),
                     __shfl_up_sync(0xffffffffu, v.z, o), __shfl_up_sync(0xffffffffu, v.w, o));
  };
  int4 ix = x, iy = y;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int4 px = shfl_up4(ix, o), py = shfl_up4(iy, o);
    if (lane >= o) {
      ix = add4(ix, px);
      iy = add4(iy, py);
    }
  }
  if (lane == 31) {
    sx[warp] = ix;
    sy[warp] = iy;
  }
  __syncthreads();
  if (warp == 0) {
    const int4 z = make_int4(0, 0, 0, 0);
    const int4 wx = lane < nw ? sx[lane] : z, wy = lane < nw ? sy[lane] : z;
    int4 jx = wx, jy = wy;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int4 px = shfl_up4(jx, o), py = shfl_up4(jy, o);
      if (lane >= o) {
        jx = add4(jx, px);
        jy = add4(jy, py);
      }
    }
    sx[lane] = sub4(jx, wx);  // exclusive
    sy[lane] = sub4(jy, wy);
    if (lane == 31) {
      sx[32] = jx;
      sy[32] = jy;
    }
  }
  __syncthreads();
  *ox = add4(sx[warp], sub4(ix, x));
  *oy = add4(sy[warp], sub4(iy, y));
  *tx = sx[32];
  *ty = sy[32];
  __syncthreads();
}

// Last index i in [0, n) with off[i] <= x: the request that owns entry x
// when off[] holds the exclusive prefix sums of per-request counts.
__device__ __forceinline__ int find_owner(const int* off, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

struct ReqInfo {
  int kind;  // 0 nothing, 1 decode, 2 prefill
  int n, L, q0;
  int bad;   // PKV_DEV_ERR_* bits of a request that fails a check
};

__device__ ReqInfo classify(const AttnArgs& a, int r) {
  ReqInfo ri{0, 0, 0, 0, 0};
  const int q0 = __ldcg(a.qsl + r), q1 = __ldcg(a.qsl + r + 1), L = __ldcg(a.seq_lens + r);
  int bad = 0;
  if (q0 < 0 || q1 < q0 || (int64_t)q1 > a.q_rows)
    bad = PKV_DEV_ERR_QSL;
  else if (L < 0 || L < q1 - q0)
    bad = PKV_DEV_ERR_SEQ_LEN;
  else if (((int64_t)L + kBlockSize - 1) / kBlockSize > a.bt_width)
    bad = PKV_DEV_ERR_BT_WIDTH;
  if (bad) {
    ri.bad = bad;
    return ri;
  }
  ri.n = q1 - q0;
  ri.L = L;
  ri.q0 = q0;
  // decode: the query tokens x heads of a KV head fit one decode unit's rows
  // (speculative / multi-token decode included); prefill: anything longer
  const int G = a.hq / a.hkv;
  ri.kind = ri.n == 0 ? 0 : (ri.n * G <= dec_rows_cap(G) ? 1 : 2);
  if (ri.kind == 2 && a.kv_int8) {  // int8 caches are read by the decode path only
    ri.kind = 0;
    ri.bad = PKV_DEV_ERR_INT8_PREFILL;
  }
  return ri;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(AttnArgs a, Workspace ws,
                                                            int dec_grid) {
  __shared__ int4 smem33[33], smem33b[33];
  __shared__ long long red[32];
  const int tid = threadIdx.x, nt = blockDim.x, nw = nt >> 5;
  // Let the decode grid set up at once.  The metadata is read before the
  // wait for the kernel before this one: that kernel let this grid start
  // either by finishing, or, as this library's cache write, after its own
  // wait for everything before it (it does not touch the metadata), or, as
  // another plan kernel (pkv_plan), without writing the metadata.  The wait
  // comes before the first write to the workspace (which that plan kernel
  // may still be writing, or the previous step's kernels still reading), and
  // this grid does not finish before it: a kernel that waits for this one
  // also finds the cache write done.
  grid_dep_launch();

  // pass 1: total decode keys, decode requests and their longest length, to
  // size the split-KV chunk (a thread keeps its first request's
  // classification for pass 2)
  long long dec_keys = 0;
  int dec_reqs = 0, dec_lmax = 0, dec_rmax = 0;  // rmax: most query rows of a decode
  int pre_tiles = 0, pre_max = 0;  // key tiles of the prefill entries: sum, longest
  ReqInfo first{0, 0, 0, 0, 0};
  for (int r = tid; r < a.num_reqs; r += nt) {
    ReqInfo ri = classify(a, r);
    if (r == tid) first = ri;
    if (ri.kind == 1) {
      dec_keys += ri.L;
      dec_reqs += 1;
      dec_lmax = max(dec_lmax, ri.L);
      dec_rmax = max(dec_rmax, ri.n * (a.hq / a.hkv));
    } else if (ri.kind == 2) {
      // query tile t (rows up to min(128 (t + 1), n)) reads ctx + its last row
      // keys; the last tile reads them all
      const int ctx = ri.L - ri.n;
      for (int t = 0; t * kPreTileQ < ri.n; ++t)
        pre_tiles += (ctx + min(kPreTileQ * (t + 1), ri.n) + kPreTileQ - 1) / kPreTileQ;
      pre_max = max(pre_max, (ri.L + kPreTileQ - 1) / kPreTileQ);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    dec_keys += __shfl_xor_sync(0xffffffffu, dec_keys, o);
    dec_reqs += __shfl_xor_sync(0xffffffffu, dec_reqs, o);
    dec_lmax = max(dec_lmax, __shfl_xor_sync(0xffffffffu, dec_lmax, o));
    dec_rmax = max(dec_rmax, __shfl_xor_sync(0xffffffffu, dec_rmax, o));
    pre_tiles += __shfl_xor_sync(0xffffffffu, pre_tiles, o);
    pre_max = max(pre_max, __shfl_xor_sync(0xffffffffu, pre_max, o));
  }
  __shared__ int red_n[32], red_l[32], red_r[32], red_t[32], red_m[32];
  if ((tid & 31) == 0) {
    red[tid >> 5] = dec_keys;
    red_n[tid >> 5] = dec_reqs;
    red_l[tid >> 5] = dec_lmax;
    red_r[tid >> 5] = dec_rmax;
    red_t[tid >> 5] = pre_tiles;
    red_m[tid >> 5] = pre_max;
  }
  __syncthreads();
  if (tid < 32) {
    long long x = tid < nw ? red[tid] : 0;
    int n = tid < nw ? red_n[tid] : 0, l = tid < nw ? red_l[tid] : 0;
    int rr = tid < nw ? red_r[tid] : 0;
    int pt = tid < nw ? red_t[tid] : 0, pm = tid < nw ? red_m[tid] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      x += __shfl_xor_sync(0xffffffffu, x, o);
      n += __shfl_xor_sync(0xffffffffu, n, o);
      l = max(l, __shfl_xor_sync(0xffffffffu, l, o));
      rr = max(rr, __shfl_xor_sync(0xffffffffu, rr, o));
      pt += __shfl_xor_sync(0xffffffffu, pt, o);
      pm = max(pm, __shfl_xor_sync(0xffffffffu, pm, o));
    }
    if (tid == 0) {
      red[0] = x;
      red_n[0] = n;
      red_l[0] = l;
      red_r[0] = rr;
      red_t[0] = pt;
      red_m[0] = pm;
    }
  }
  __syncthreads();
  const long long total_keys = red[0];
  const long long dec_pairs = (long long)red_n[0] * a.hkv;  // (request, KV head) pairs
  const int lmax = red_l[0];
  const int rmax = red_r[0];
  // aim for about four units per decode worker (dec_grid = workers), in
  // whole 64-key tiles, at most kMaxChunk keys; at least kMinChunk keys, and
  // at least 32 keys per query head of the group, so that a split's partial
  // result (G rows of 130 fp32) stays small next to the K/V bytes it read
  // (32-bit divisions below: a 64-bit one is a long software sequence, on
  // this kernel's critical path.  The key total is saturated just past the
  // largest chunk times the divisor and the capacities at INT_MAX, which
  // changes no result: past those bounds the clamp to kMaxChunk, or the
  // smaller per-pair count, decides.)
  const unsigned den = 4u * (unsigned)dec_grid;  // dec_grid: a few thousand workers at most
  const long long tk = total_keys * a.hkv;
  unsigned want = tk > (long long)kMaxChunk * den ? (unsigned)kMaxChunk + 1u
                                                  : ((unsigned)tk + den - 1u) / den;
  want = (want + kDecTile - 1) / kDecTile * kDecTile;
  const int G = a.hq / a.hkv;
  const int lo_chunk = max(kMinChunk, 32 * G);
  int chunk = want < (unsigned)lo_chunk ? lo_chunk : (want > (unsigned)kMaxChunk ? kMaxChunk : (int)want);
  // When even the longest request's splits, times the pairs, fit one wave of
  // workers, the step takes one unit's time: give every pair as many splits
  // as the wave has room for (units of at most that many keys), so that the
  // wave is full and each unit short.  The workspace is sized for chunks of
  // kMinChunk keys; a shorter chunk, down to one 64-key tile, is taken where
  // the workspace also holds the units and partial rows it makes: at most
  // `per` splits a pair, pairs x per units and pairs x per x rmax rows.  (The
  // batch is small then: the extra partial results are small next to the
  // latency a long unit's chain of pages costs.)  A chunk of kMinChunk keys
  // or more is cut here at whole pages (all the decode kernels need), so that
  // the units come as close to one per worker as the lengths allow (32 MQA
  // requests of 32,769 keys on 1216 int8 workers: 1216 units of 864 keys
  // instead of 1184 of 896, 2% faster).  In both branches the pairs are at
  // most the workers.
  auto page_chunk = [](unsigned c) {
    const unsigned p = (c + kBlockSize - 1) / kBlockSize * kBlockSize;
    return p < (unsigned)kMinChunk ? (unsigned)kMinChunk : p;
  };
  if (dec_pairs > 0 && dec_pairs * ((lmax + chunk - 1) / chunk) <= dec_grid) {
    const unsigned pairs = (unsigned)dec_pairs;
    const unsigned per_pair = (unsigned)dec_grid / pairs;
    const unsigned c1 = ((unsigned)lmax + per_pair - 1u) / per_pair;
    unsigned c = (c1 + kDecTile - 1) / kDecTile * kDecTile;
    if (c >= (unsigned)kMinChunk) {
      c = page_chunk(c1);
    } else {
      const unsigned mu = (unsigned)min(ws.max_units, (int64_t)INT_MAX);
      const unsigned mp = (unsigned)min(ws.max_part_rows, (int64_t)INT_MAX);
      unsigned per = per_pair;
      per = min(per, mu / pairs);
      per = min(per, mp / (pairs * (unsigned)max(rmax, 1)));
      unsigned c2 = per >= 1u ? ((unsigned)lmax + per - 1u) / per : (unsigned)kMinChunk;
      c2 = (c2 + kDecTile - 1) / kDecTile * kDecTile;
      c = c2 < (unsigned)kMinChunk ? (c2 > c ? c2 : c) : (unsigned)kMinChunk;
    }
    if ((int)c < chunk) chunk = (int)c;
  } else if (dec_pairs > 0 && dec_pairs <= dec_grid) {
    // More splits than one wave of workers, but every pair fits in it with
    // a somewhat longer chunk: one wave of units under twice as long beats
    // two waves (32 MQA requests of 32,769 keys on 912 workers: 1216-key
    // units, 864 of them, instead of 1056 units of 1024 keys).  Whole 64-key
    // tiles here: 896 units of 1184 keys kept more SMs at six busy worker
    // pairs and ran 2.6% slower.
    const unsigned per_pair = (unsigned)dec_grid / (unsigned)dec_pairs;
    unsigned c = ((unsigned)lmax + per_pair - 1u) / per_pair;
    c = (c + kDecTile - 1) / kDecTile * kDecTile;
    if (c <= (unsigned)kMaxChunk && (int)c < 2 * chunk) chunk = (int)c;
  }

  // Units are listed roughly longest first, in five classes: every request's
  // full chunks, then the last (shorter) pieces by the quarter of a chunk
  // they fill, longest first, so that the tail of the dynamic schedule is
  // made of short units.  cls_base[c] = first unit of class c.
  auto last_class = [&](int L) {  // 0: no last piece; 1..4 longest to shortest
    const int rem = L % chunk;
    return rem == 0 ? 0 : 4 - min(3, (rem - 1) * 4 / chunk);
  };
  int4 cnt = make_int4(0, 0, 0, 0);  // units of classes 0..3 of this thread's requests
                                     // (class 4 comes last: its count is not needed)
  for (int r = tid; r < a.num_reqs; r += nt) {
    const ReqInfo ri = r == tid ? first : classify(a, r);
    if (ri.kind != 1) continue;
    cnt.x += (ri.L / chunk) * a.hkv;
    const int c = last_class(ri.L);
    if (c == 1) cnt.y += a.hkv;
    if (c == 2) cnt.z += a.hkv;
    if (c == 3) cnt.w += a.hkv;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cnt.x += __shfl_xor_sync(0xffffffffu, cnt.x, o);
    cnt.y += __shfl_xor_sync(0xffffffffu, cnt.y, o);
    cnt.z += __shfl_xor_sync(0xffffffffu, cnt.z, o);
    cnt.w += __shfl_xor_sync(0xffffffffu, cnt.w, o);
  }
  if ((tid & 31) == 0) smem33[tid >> 5] = cnt;
  __syncthreads();
  int4 cls = make_int4(0, 0, 0, 0);
#pragma unroll 4
  for (int w = 0; w < nw; ++w) {  // (every thread, the same order)
    const int4 v = smem33[w];
    cls.x += v.x;
    cls.y += v.y;
    cls.z += v.z;
    cls.w += v.w;
  }
  __syncthreads();  // smem33 is reused by the scans
  const int cls_base[5] = {0, cls.x, cls.x + cls.y, cls.x + cls.y + cls.z,
                           cls.x + cls.y + cls.z + cls.w};

  // pass 2: per-request offsets (block scans), then the work lists written
  // cooperatively: consecutive threads write consecutive entries, each
  // finding its request by binary search over the chunk's offsets
  __shared__ int s_off_u[kPlanThreads + 1], s_off_t[kPlanThreads + 1], s_off_q[kPlanThreads + 1];
  __shared__ int s_off_f[kPlanThreads], s_off_l[kPlanThreads];  // full chunks, last piece
  __shared__ int s_off_p[kPlanThreads], s_len[kPlanThreads], s_n[kPlanThreads];
  __shared__ int s_q0[kPlanThreads];
  __shared__ int s_max_rows;
  if (tid == 0) s_max_rows = 0;
  __syncthreads();
  int unit_carry = 0, part_carry = 0, pre_carry = 0, pair_carry = 0;
  int cls_carry[5] = {0, 0, 0, 0, 0};
  for (int base = 0; base < a.num_reqs; base += nt) {
    const int r = base + tid;
    ReqInfo ri{0, 0, 0, 0, 0};
    if (r < a.num_reqs) ri = base == 0 ? first : classify(a, r);
    if (ri.bad && blockIdx.x == 0) atomicOr(ws.err, ri.bad);
    int units = 0, parts = 0, tiles = 0, pairs = 0, fulls = 0, lcls = 0;
    if (ri.kind == 1) {
      const int nsplit = (ri.L + chunk - 1) / chunk;
      units = nsplit * a.hkv;
      fulls = (ri.L / chunk) * a.hkv;
      lcls = last_class(ri.L);
      parts = nsplit > 1 ? units * ri.n * G : 0;  // partial rows
      pairs = nsplit > 1 ? a.hkv : 0;
      if (nsplit > 1) atomicMax(&s_max_rows, ri.n * G);
    } else if (ri.kind == 2) {
      tiles = (ri.n + kPreTileQ - 1) / kPreTileQ;
    }
    // the per-request offsets, and those inside the classes: full chunks and
    // the last piece's class 1..3; a request's units are its full chunks and
    // its last piece (class 1..4), so class 4's offsets are what remains
    const int lu = units - fulls;  // a.hkv or 0
    int4 off, off2, tot, tot2;
    block_exclusive_scan8(make_int4(units, parts, tiles, pairs),
                          make_int4(fulls, lcls == 1 ? lu : 0, lcls == 2 ? lu : 0, lcls == 3 ? lu : 0),
                          &off, &off2, &tot, &tot2, smem33, smem33b);
    const int off_u = off.x, off_p = off.y, off_t = off.z, off_q = off.w;
    const int tot_u = tot.x, tot_p = tot.y, tot_t = tot.z, tot_q = tot.w;
    const int off4 = off_u - (off2.x + off2.y + off2.z + off2.w);
    const int tot4 = tot_u - (tot2.x + tot2.y + tot2.z + tot2.w);
    s_off_f[tid] = cls_base[0] + cls_carry[0] + off2.x;
    {
      const int ofs = lcls == 1 ? off2.y : (lcls == 2 ? off2.z : (lcls == 3 ? off2.w : off4));
      s_off_l[tid] = lcls == 0 ? 0 : cls_base[lcls] + cls_carry[lcls] + ofs;
    }
    s_off_u[tid] = off_u;
    s_off_t[tid] = off_t;
    s_off_q[tid] = off_q;
    s_off_p[tid] = part_carry + off_p;
    s_len[tid] = ri.L;
    s_n[tid] = ri.n;
    s_q0[tid] = ri.q0;
    if (tid == 0) {
      s_off_u[nt] = tot_u;
      s_off_t[nt] = tot_t;
      s_off_q[nt] = tot_q;
    }
    if (base == 0) grid_dep_wait();  // the first write to the workspace follows
    __syncthreads();
    // decode units and split pairs: one warp of the grid per request (a
    // request's entries are contiguous), lanes over its entries, so that
    // consecutive lanes write consecutive entries with no search for the owner
    for (int lo = blockIdx.x * nw + (tid >> 5); lo < nt && base + lo < a.num_reqs;
         lo += gridDim.x * nw) {
      const int ln = tid & 31;
      const int cnt_u = s_off_u[lo + 1] - s_off_u[lo];
      if (cnt_u == 0) continue;
      const int L = s_len[lo], qn = s_n[lo];
      const int nsplit = (L + chunk - 1) / chunk, nfull = L / chunk;
      for (int rem = ln; rem < cnt_u; rem += 32) {
        const int sp = rem / a.hkv, g = rem - sp * a.hkv;
        const int64_t idx = sp < nfull ? (int64_t)s_off_f[lo] + rem : (int64_t)s_off_l[lo] + g;
        if (idx >= ws.max_units) break;
        // two 16-byte stores per unit
        int4* dst = reinterpret_cast<int4*>(ws.units + idx);
        dst[0] = make_int4(base + lo, g | (qn << 16), L - qn, nsplit);
        dst[1] = make_int4(sp * chunk, min(L, (sp + 1) * chunk),
                           nsplit > 1 ? s_off_p[lo] + (g * nsplit + sp) * qn * G : -1, s_q0[lo]);
      }
      const int cnt_q = s_off_q[lo + 1] - s_off_q[lo];
      for (int g = ln; g < cnt_q; g += 32) {
        const int64_t idx = (int64_t)pair_carry + s_off_q[lo] + g;
        if (idx >= ws.max_pairs) break;
        int4* dst = reinterpret_cast<int4*>(ws.pairs + idx);
        dst[0] = make_int4(base + lo, g, s_off_p[lo] + g * nsplit * qn * G, nsplit);
        dst[1] = make_int4(s_q0[lo], qn, 0, 0);
      }
    }
    for (int i = blockIdx.x * nt + tid; i < tot_t; i += gridDim.x * nt) {
      const int lo = find_owner(s_off_t, nt, i);
      // a request's query tiles from the last (most keys) to the first, so
      // that the persistent prefill grid starts with the longest items
      const int n = s_n[lo], ctx = s_len[lo] - n;
      const int t = (n + kPreTileQ - 1) / kPreTileQ - 1 - (i - s_off_t[lo]);
      const int64_t idx = (int64_t)pre_carry + i;
      if (idx >= ws.max_pre) break;
      const int last_row = min(kPreTileQ * (t + 1), n);
      int4* dst = reinterpret_cast<int4*>(ws.pre + idx);
      dst[0] = make_int4(base + lo, t, (ctx + last_row + kPreTileQ - 1) / kPreTileQ, s_q0[lo]);
      dst[1] = make_int4(n, s_len[lo], 0, 0);
    }
    unit_carry += tot_u;
    cls_carry[0] += tot2.x;
    cls_carry[1] += tot2.y;
    cls_carry[2] += tot2.z;
    cls_carry[3] += tot2.w;
    cls_carry[4] += tot4;
    part_carry += tot_p;
    pre_carry += tot_t;
    pair_carry += tot_q;
    __syncthreads();  // the chunk's offsets are reused by the next chunk
  }
  grid_dep_wait();  // (already returned unless the loop above ran no chunk)
  if (blockIdx.x == 0 && tid == 0) {
    // A plan that does not fit the workspace runs nothing: entries past a
    // capacity were not written and partial rows past it have no room, so
    // the whole step is dropped (no output row is written) and reported.
    // The host sizes the workspace so that this cannot happen.
    const bool fits = (int64_t)unit_carry <= ws.max_units && (int64_t)pre_carry <= ws.max_pre &&
                      (int64_t)pair_carry <= ws.max_pairs &&
                      (int64_t)part_carry <= ws.max_part_rows;
    if (!fits) atomicOr(ws.err, PKV_DEV_ERR_CAPACITY);
    ws.hdr->n_dec_units = fits ? unit_carry : 0;
    ws.hdr->n_pre_entries = fits ? pre_carry : 0;
    ws.hdr->dec_counter = 0;
    ws.hdr->pre_counter = 0;
    ws.hdr->chunk = chunk;
    ws.hdr->n_pairs = fits ? pair_carry : 0;
    ws.hdr->max_rows = s_max_rows;
    ws.hdr->pre_tiles = red_t[0];
    ws.hdr->pre_max_tiles = red_m[0];
  }
}

}  // namespace

cudaError_t launch_plan(const AttnArgs& a, const Workspace& ws, int dec_grid, cudaStream_t st) {
  // a thread per request of a chunk (whole warps, at most 1024); one warp
  // of the grid per request of the first chunk, at most 16 CTAs
  const int threads = std::min(kPlanThreads, std::max(32, (a.num_reqs + 31) / 32 * 32));
  const int warps = threads / 32;
  const int want = (std::min(a.num_reqs, threads) + warps - 1) / warps;
  const int grid = std::max(1, std::min(16, want));
  return launch_dependent(plan_kernel, dim3(grid), dim3(threads), 0, st, a, ws, dec_grid);
}

}  // namespace pkv
