// The merge of split-KV decode results, run after the decode kernel: by every
// warp of the prefill kernel's launch at its end (bf16 calls), by the combine
// kernel (int8 calls).
#pragma once

#include "pkv_device.cuh"

namespace pkv {
namespace dev {

// Merge of split results: one (split pair, query row) per warp (warp_id of
// n_warps in the grid), four output columns per lane, the splits merged in
// one pass with the online-softmax identity the decode loop uses between
// pages (a running max M; the sum and the output so far are scaled by
// exp2(M_old - M_new) when it grows).  A
// split that saw no key of the row (m = -inf: only later splits of a
// multi-token row) contributes nothing; the first split always holds key 0.
// Rows are (query token, head in group); pairs with fewer rows than the
// largest skip the rest.
__device__ __forceinline__ void combine_splits(const AttnArgs& a, const Workspace& ws, int warp_id,
                                               int n_warps) {
  const int G = a.hq / a.hkv;
  // (the plan's lists are read through L2: the plan kernel ran two launches
  // before this one)
  const int max_rows = __ldcg(&ws.hdr->max_rows);
  const int n_items = __ldcg(&ws.hdr->n_pairs) * max_rows;
  const int lane = threadIdx.x & 31;
  for (int item = warp_id; item < n_items; item += n_warps) {
    const int4 pw0 = __ldcg(reinterpret_cast<const int4*>(ws.pairs + item / max_rows));
    const int4 pw1 = __ldcg(reinterpret_cast<const int4*>(ws.pairs + item / max_rows) + 1);
    const SplitPair sp{pw0.x, pw0.y, pw0.z, pw0.w, pw1.x, pw1.y, pw1.z, pw1.w};
    const int row = item % max_rows;
    const int q0 = sp.q0;
    const int rows = sp.qn * G;
    if (row >= rows) continue;
    const float* ml = ws.part_ml + ((int64_t)sp.first + row) * 2;
    const float* po = ws.part_o + ((int64_t)sp.first + row) * kHeadSize + 4 * lane;
    float M = -INFINITY, lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int s = 0; s < sp.nsplit; ++s) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(ml + (int64_t)s * rows * 2));
      const float4 o = __ldcg(reinterpret_cast<const float4*>(po + (int64_t)s * rows * kHeadSize));
      const float Mn = fmaxf(M, v.x);
      const float fo = M == -INFINITY ? 0.f : fast_exp2(M - Mn);
      const float fn = v.x == -INFINITY ? 0.f : fast_exp2(v.x - Mn);
      lsum = lsum * fo + v.y * fn;
      acc.x = acc.x * fo + o.x * fn;
      acc.y = acc.y * fo + o.y * fn;
      acc.z = acc.z * fo + o.z * fn;
      acc.w = acc.w * fo + o.w * fn;
      M = Mn;
    }
    const float inv = 1.f / lsum;
    uint16_t* orow = a.out + (int64_t)(q0 + row / G) * a.out_stride +
                     (int64_t)(sp.g * G + row % G) * kHeadSize + 4 * lane;
    *reinterpret_cast<uint2*>(orow) =
        make_uint2(pack_bf16(acc.x * inv, acc.y * inv), pack_bf16(acc.z * inv, acc.w * inv));
  }
}

}  // namespace dev
}  // namespace pkv
