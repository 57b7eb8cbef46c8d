// Step-side metadata: positions, seq_lens, the gathered block table and the
// slot of every scheduled token, from the request state on the device.
//
// "Tour: One forward pass", stop 3 (prepare_pos_seq_lens): token t of request
// r sits at num_computed[r] + (t - query_start_loc[r]); seq_len = num_computed
// + query_len.  Stop 4 (gather_block_tables): the persistent block-table row of
// each request's slot (idx_mapping) is copied into batch order.  Stop 4
// (compute_slot_mappings): slot = block_number * block_size + offset, and the
// rows past the last request's tokens get PAD_SLOT_ID = -1.  The padding rows
// of positions are not written (stop 3).
//
// One launch does all three: threads over token rows (positions and slots, the
// request found by binary search over query_start_loc, which is short and
// L2-resident), over request x block-table column (the gather), and over
// requests (seq_lens).  Everything is integer work bound by launch latency.
#include "pkv_internal.cuh"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256) prepare_kernel(PrepArgs p) {
  const int64_t T = p.num_tokens_padded;
  const int64_t gather = (int64_t)p.num_reqs * p.bt_width;
  const int64_t total = T + gather + p.num_reqs;
  const int64_t ntok = p.num_reqs > 0 ? p.qsl[p.num_reqs] : 0;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < T) {
      const int64_t t = i;
      if (t >= ntok) {  // padding row
        p.slot_mapping[t] = -1;
        continue;
      }
      int lo = 0, hi = p.num_reqs - 1;  // last r with qsl[r] <= t
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.qsl[mid] <= t) lo = mid; else hi = mid - 1;
      }
      const int r = lo;
      const int row = p.idx ? p.idx[r] : r;
      const int64_t pos = (int64_t)p.num_computed[r] + (t - p.qsl[r]);
      p.positions[t] = pos;
      const int64_t bi = pos / kBlockSize;
      if (row < 0 || row >= p.pbt_rows || bi >= p.bt_width || pos < 0) {
        atomicOr(p.err, PKV_DEV_ERR_BT_WIDTH);
        p.slot_mapping[t] = -1;
        continue;
      }
      const int32_t blk = p.pbt[(int64_t)row * p.bt_width + bi];
      p.slot_mapping[t] = (int64_t)blk * kBlockSize + pos % kBlockSize;
    } else if (i < T + gather) {
      const int64_t k = i - T;
      const int r = (int)(k / p.bt_width);
      const int64_t b = k - (int64_t)r * p.bt_width;
      const int row = p.idx ? p.idx[r] : r;
      if (p.block_table)
        p.block_table[k] = (row >= 0 && row < p.pbt_rows) ? p.pbt[(int64_t)row * p.bt_width + b]
                                                          : -1;
    } else {
      const int r = (int)(i - T - gather);
      p.seq_lens[r] = p.num_computed[r] + (p.qsl[r + 1] - p.qsl[r]);
    }
  }
}

}  // namespace

cudaError_t launch_prepare(const PrepArgs& p, int sms, cudaStream_t st) {
  const int64_t total = p.num_tokens_padded + (int64_t)p.num_reqs * p.bt_width + p.num_reqs;
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sms * 8) blocks = (int64_t)sms * 8;
  if (blocks < 1) blocks = 1;
  prepare_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
