// Per-query top-k of the index scores: an exact block-wide radix select.
//
// ("DeepSeek3.2: Onboard sparse attention", Background: top-k token selection
// per query turns the index scores into the index mask. Equal scores go to the
// lower key index, -0.0 equals +0.0.)
//
// One CTA per query row (b, t). The valid keys are s in [0, t] with, when
// segment ids are given, seg[s] == seg[t]; n = their number.
//   n <= k : every valid key is selected (ordered compaction, no score read).
//   n >  k : the scores are mapped to order-preserving 32-bit keys (-0 -> +0),
//            staged in shared memory when the row fits, and the k-th largest
//            key T is found digit by digit (4 x 8 bits, warp-aggregated
//            shared-memory histograms via __match_any_sync). A final ordered
//            pass selects every key > T and the lowest-index `need` keys == T,
//            writing positions from one block-wide scan, so the output is
//            ascending. Slots m..k-1 get -1.
// Rows longer than the shared-memory stage are re-read from global memory
// (L2) on every digit pass.

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kStageMax = 16384;   // keys staged in shared memory per row

struct TopkParams {
  const float* scores;
  long long ld;
  const int32_t* seg;
  int B, S, k;
  int32_t* idx;
  int32_t* count;
  int stage_cap;
};

struct TopkSmem {
  uint32_t hist[256];
  int warp_tot[kWarps];
  int bcast[4];
};

// Larger float -> larger key; -0.0 and +0.0 map to the same key; key 0 is never
// produced by a non-NaN score and marks an invalid (masked) key.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Inclusive block scan of one int per thread; returns the inclusive value and
// the block total.
__device__ __forceinline__ int block_scan(int v, int& total, TopkSmem* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm->warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < kWarps ? sm->warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < kWarps) sm->warp_tot[lane] = w;   // inclusive prefix of warp totals
  }
  __syncthreads();
  const int before = warp > 0 ? sm->warp_tot[warp - 1] : 0;
  total = sm->warp_tot[kWarps - 1];
  __syncthreads();   // warp_tot is reused by the next call
  return x + before;
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkSmem* sm = reinterpret_cast<TopkSmem*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + sizeof(TopkSmem));

  // long rows first
  const long long row = static_cast<long long>(gridDim.x) - 1 - blockIdx.x;
  const int b = static_cast<int>(row / p.S);
  const int t = static_cast<int>(row - static_cast<long long>(b) * p.S);
  const int len = t + 1;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int32_t* seg_row = p.seg ? p.seg + static_cast<long long>(b) * p.S : nullptr;
  const int seg_t = seg_row ? seg_row[t] : 0;
  const float* srow = p.scores + row * p.ld;
  int32_t* out = p.idx + row * p.k;

  // number of valid keys
  int n = len;
  if (seg_row) {
    int c = 0;
    for (int s = tid; s < len; s += kThreads) c += (seg_row[s] == seg_t);
    int tot;
    block_scan(c, tot, sm);
    n = tot;
  }

  if (n <= p.k) {
    // every valid key is selected, in ascending order
    int base = 0;
    for (int s0 = 0; s0 < len; s0 += kThreads) {
      const int s = s0 + tid;
      const int v = (s < len) && (!seg_row || seg_row[s] == seg_t);
      int tot;
      const int incl = block_scan(v, tot, sm);
      if (v) out[base + incl - 1] = s;
      base += tot;
    }
    for (int j = n + tid; j < p.k; j += kThreads) out[j] = -1;
    if (p.count && tid == 0) p.count[row] = n;
    return;
  }

  const bool staged = len <= p.stage_cap;
  if (staged) {
    for (int s = tid; s < len; s += kThreads) {
      const bool v = !seg_row || seg_row[s] == seg_t;
      keys[s] = v ? order_key(__ldg(srow + s)) : 0u;
    }
  }
  __syncthreads();

  auto key_at = [&](int s) -> uint32_t {
    if (staged) return keys[s];
    const bool v = !seg_row || seg_row[s] == seg_t;
    return v ? order_key(__ldg(srow + s)) : 0u;
  };

  // ---- radix select: the k-th largest key, 8 bits at a time
  uint32_t prefix = 0u, mask = 0u;
  int need = p.k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    if (tid < 256) sm->hist[tid] = 0u;
    __syncthreads();
    for (int s0 = 0; s0 < len; s0 += kThreads) {
      const int s = s0 + tid;
      const uint32_t key = s < len ? key_at(s) : 0u;
      const bool part = key != 0u && (key & mask) == prefix;
      const uint32_t bin = (key >> shift) & 255u;
      const uint32_t peers = __match_any_sync(0xffffffffu, part ? bin : 0xFFFFFFFFu);
      if (part && lane == __ffs(peers) - 1) atomicAdd(&sm->hist[bin], __popc(peers));
    }
    __syncthreads();
    // bins in descending order: thread i owns bin 255 - i
    int cnt = tid < 256 ? static_cast<int>(sm->hist[255 - tid]) : 0;
    int tot;
    const int incl = block_scan(cnt, tot, sm);
    if (tid < 256 && incl >= need && incl - cnt < need) {
      sm->bcast[0] = 255 - tid;      // selected bin
      sm->bcast[1] = incl - cnt;     // keys in higher bins
      sm->bcast[2] = cnt;
    }
    __syncthreads();
    const uint32_t sel = static_cast<uint32_t>(sm->bcast[0]);
    need -= sm->bcast[1];
    const int in_bin = sm->bcast[2];
    __syncthreads();
    prefix |= sel << shift;
    mask |= 255u << shift;
    if (in_bin == need) break;   // every key with this prefix is taken
  }

  // ---- ordered selection: key > T, or key == T among the first `need` of them
  int gt_base = 0, eq_base = 0;
  for (int s0 = 0; s0 < len; s0 += kThreads) {
    const int s = s0 + tid;
    const uint32_t key = s < len ? key_at(s) : 0u;
    const uint32_t km = key & mask;
    const int gt = key != 0u && km > prefix;
    const int eq = key != 0u && km == prefix;
    int tot;
    const int incl = block_scan(gt | (eq << 16), tot, sm);
    const int gt_before = gt_base + ((incl & 0xFFFF) - gt);
    const int eq_before = eq_base + ((incl >> 16) - eq);
    const int pos = gt_before + min(eq_before, need);
    if ((gt || (eq && eq_before < need)) && pos < p.k) out[pos] = s;
    gt_base += tot & 0xFFFF;
    eq_base += tot >> 16;
  }
  if (p.count && tid == 0) p.count[row] = p.k;   // n > k: exactly k selected, no padding
}

}  // namespace

int launch_topk(const float* scores, int64_t ld, const int32_t* seg, int B, int S, int k,
                int32_t* idx, int32_t* count, cudaStream_t stream) {
  TopkParams p;
  p.scores = scores;
  p.ld = ld;
  p.seg = seg;
  p.B = B;
  p.S = S;
  p.k = k;
  p.idx = idx;
  p.count = count;
  p.stage_cap = S < kStageMax ? S : kStageMax;
  const size_t smem = sizeof(TopkSmem) + static_cast<size_t>(p.stage_cap) * 4;
  if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  const long long rows = static_cast<long long>(B) * S;
  if (rows > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
  topk_kernel<<<static_cast<unsigned>(rows), kThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
