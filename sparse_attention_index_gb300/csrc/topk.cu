// Per-query top-k of the index scores: an exact block-wide radix select.
//
// ("DeepSeek3.2: Onboard sparse attention", Background: top-k token selection
// per query turns the index scores into the index mask. Equal scores go to the
// lower key index, -0.0 equals +0.0.)
//
// One CTA per query row (b, t). The valid keys are s in [0, t] with, when
// segment ids are given, seg[s] == seg[t]; n = their number.
//   n <= k : every valid key is selected (ordered compaction, no score read).
//   n >  k : the scores are mapped to order-preserving 32-bit keys (-0 -> +0)
//            and the k-th largest key T is found digit by digit with
//            shared-memory histograms. Rows that fit in shared memory are staged
//            there (16-byte asynchronous copies) and the first 11-bit histogram is
//            built while the keys are converted; at most two more levels (11, 10
//            bits) run on the staged keys, four keys per thread, and stop as soon
//            as the selected bin holds exactly the keys still needed. The final
//            ordered pass selects every key > T and the lowest-index `need` keys
//            == T: each warp owns a contiguous segment, a count sweep gives the
//            segment offsets and a write sweep places the keys, through a shared
//            staging row for coalesced stores. Longer rows take 4 x 8-bit passes
//            over global memory (L2) with warp-aggregated (__match_any_sync)
//            histograms. Slots m..k-1 get -1.

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
  uint32_t hist[2048];
  int warp_tot[kWarps];
  int wgt[kWarps], weq[kWarps];
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

// Ordered selection: for s in [0, len), flags(s) gives (gt, eq). Every gt element
// and the first `need` eq elements (in s order) are written to out[] in ascending s;
// an element's slot is (#gt before it) + min(#eq before it, need). Each warp owns one
// contiguous, 32-aligned segment; one block barrier orders the warps.
template <class Flags>
__device__ __forceinline__ void ordered_select(int len, Flags flags, int need, int32_t* out,
                                               int kmax, TopkSmem* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg_len = ((len + kThreads - 1) / kThreads) * 32;
  const int s_begin = warp * seg_len, s_end = min(len, s_begin + seg_len);
  int cg = 0, ce = 0;
  for (int s = s_begin + lane; s < s_end; s += 32) {
    const int2 f = flags(s);
    cg += f.x;
    ce += f.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cg += __shfl_xor_sync(0xffffffffu, cg, o);
    ce += __shfl_xor_sync(0xffffffffu, ce, o);
  }
  if (lane == 0) {
    sm->wgt[warp] = cg;
    sm->weq[warp] = ce;
  }
  __syncthreads();
  int gt_base = 0, eq_base = 0;
  for (int w = 0; w < warp; ++w) {
    gt_base += sm->wgt[w];
    eq_base += sm->weq[w];
  }
  const uint32_t lt = (1u << lane) - 1u;
  for (int s0 = s_begin; s0 < s_end; s0 += 32) {
    const int s = s0 + lane;
    const int2 f = s < s_end ? flags(s) : make_int2(0, 0);
    const uint32_t bg = __ballot_sync(0xffffffffu, f.x), be = __ballot_sync(0xffffffffu, f.y);
    const int eq_before = eq_base + __popc(be & lt);
    const int pos = gt_base + __popc(bg & lt) + min(eq_before, need);
    if ((f.x || (f.y && eq_before < need)) && pos < kmax) out[pos] = s;
    gt_base += __popc(bg);
    eq_base += __popc(be);
  }
}

// Over nb histogram bins taken from the top: the bin holding the `need`-th largest
// key, the number of keys in higher bins and in that bin (broadcast through sm).
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nb, int need, TopkSmem* sm,
                                         int& bin, int& above, int& in_bin) {
  const int per = nb / kThreads;   // 4 or 2 bins per thread, highest bins to thread 0
  const int tid = threadIdx.x;
  int c[4] = {0, 0, 0, 0};
  int sum = 0;
  for (int i = 0; i < per; ++i) {
    c[i] = static_cast<int>(hist[nb - 1 - (tid * per + i)]);
    sum += c[i];
  }
  int tot;
  const int incl = block_scan(sum, tot, sm);
  int run = incl - sum;
  for (int i = 0; i < per; ++i) {
    if (run < need && run + c[i] >= need) {
      sm->bcast[0] = nb - 1 - (tid * per + i);
      sm->bcast[1] = run;
      sm->bcast[2] = c[i];
    }
    run += c[i];
  }
  __syncthreads();
  bin = sm->bcast[0];
  above = sm->bcast[1];
  in_bin = sm->bcast[2];
  __syncthreads();
}

// Final ordered selection over the staged keys (uint4 groups of four consecutive
// keys): every key with (key & mask) > prefix and the first `need` keys with
// (key & mask) == prefix, written to out[] in ascending key index. Each warp owns
// a contiguous segment of groups; a count sweep gives the segment offsets, a
// write sweep places each key at (#gt before it) + min(#eq before it, need).
__device__ __forceinline__ void select_staged(const uint4* keys4, int nq, uint32_t mask,
                                              uint32_t prefix, int need, int32_t* out,
                                              int kmax, TopkSmem* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int segq = ((nq + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int q_begin = warp * segq, q_end = min(nq, q_begin + segq);
  int cg = 0, ce = 0;
  for (int q = q_begin + lane; q < q_end; q += 32) {
    const uint4 kv = keys4[q];
    const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t km = kk[e] & mask;
      cg += (kk[e] != 0u && km > prefix);
      ce += (kk[e] != 0u && km == prefix);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    cg += __shfl_xor_sync(0xffffffffu, cg, o);
    ce += __shfl_xor_sync(0xffffffffu, ce, o);
  }
  if (lane == 0) {
    sm->wgt[warp] = cg;
    sm->weq[warp] = ce;
  }
  __syncthreads();
  int gt_base = 0, eq_base = 0;
  for (int w = 0; w < warp; ++w) {
    gt_base += sm->wgt[w];
    eq_base += sm->weq[w];
  }
  for (int q0 = q_begin; q0 < q_end; q0 += 32) {
    const int q = q0 + lane;
    uint32_t kk[4] = {0u, 0u, 0u, 0u};
    if (q < q_end) {
      const uint4 kv = keys4[q];
      kk[0] = kv.x;
      kk[1] = kv.y;
      kk[2] = kv.z;
      kk[3] = kv.w;
    }
    int fg[4], fe[4], ng = 0, ne = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t km = kk[e] & mask;
      fg[e] = kk[e] != 0u && km > prefix;
      fe[e] = kk[e] != 0u && km == prefix;
      ng += fg[e];
      ne += fe[e];
    }
    // warp inclusive scan of (gt count | eq count << 16)
    const int own = ng | (ne << 16);
    int incl = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int excl = incl - own;
    int g_before = gt_base + (excl & 0xFFFF), e_before = eq_base + (excl >> 16);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int pos = g_before + min(e_before, need);
      if ((fg[e] || (fe[e] && e_before < need)) && pos < kmax) out[pos] = 4 * q + e;
      g_before += fg[e];
      e_before += fe[e];
    }
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    gt_base += tot & 0xFFFF;
    eq_base += tot >> 16;
  }
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
    ordered_select(
        len, [&](int s) { return make_int2(!seg_row || seg_row[s] == seg_t, 0); }, 0, out, p.k,
        sm);
    for (int j = n + tid; j < p.k; j += kThreads) out[j] = -1;
    if (p.count && tid == 0) p.count[row] = n;
    return;
  }

  const bool staged = len <= p.stage_cap;
  if (staged) {
    // ---- rows held in shared memory: 11 + 11 + 10 bit radix select, the first
    // histogram built while the row is loaded
    // raw scores -> shared memory with 16-byte asynchronous copies (rows are
    // 16-byte aligned: ld is a multiple of 4)
    const int nvec = len >> 2;
    for (int c = tid; c < nvec; c += kThreads)
      cp_async_16(smem_u32(keys + 4 * c), srow + 4 * c, 16u);
    cp_async_commit();
    for (int s = 4 * nvec + tid; s < len; s += kThreads)
      keys[s] = __float_as_uint(__ldg(srow + s));
    for (int i = tid; i < 2048; i += kThreads) sm->hist[i] = 0u;
    cp_async_wait<0>();
    __syncthreads();
    // order keys in place (invalid -> 0; the tail of the last uint4 -> 0) and
    // the first 11-bit histogram, four consecutive keys per thread
    const int nq = (len + 3) >> 2;
    uint4* keys4 = reinterpret_cast<uint4*>(keys);
    for (int c = tid; c < nq; c += kThreads) {
      const uint4 raw = keys4[c];
      const uint32_t rv[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t kq[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int si = 4 * c + e;
        const bool v = si < len && (!seg_row || seg_row[si] == seg_t);
        kq[e] = v ? order_key(__uint_as_float(rv[e])) : 0u;
      }
      keys4[c] = make_uint4(kq[0], kq[1], kq[2], kq[3]);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (kq[e] != 0u) atomicAdd(&sm->hist[kq[e] >> 21], 1u);
    }
    __syncthreads();
    int bin, above, in_bin;
    find_bin(sm->hist, 2048, p.k, sm, bin, above, in_bin);
    uint32_t prefix = static_cast<uint32_t>(bin) << 21, mask = 0xFFE00000u;
    int need = p.k - above;
    const int shifts[2] = {10, 0};
    const int nbins[2] = {2048, 1024};
#pragma unroll 1
    for (int lvl = 0; lvl < 2 && in_bin != need; ++lvl) {
      const int shift = shifts[lvl], nb = nbins[lvl];
      for (int i = tid; i < nb; i += kThreads) sm->hist[i] = 0u;
      __syncthreads();
      for (int c = tid; c < nq; c += kThreads) {
        const uint4 kv = keys4[c];
        const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (kk[e] != 0u && (kk[e] & mask) == prefix)
            atomicAdd(&sm->hist[(kk[e] >> shift) & static_cast<uint32_t>(nb - 1)], 1u);
      }
      __syncthreads();
      find_bin(sm->hist, nb, need, sm, bin, above, in_bin);
      prefix |= static_cast<uint32_t>(bin) << shift;
      mask |= static_cast<uint32_t>(nb - 1) << shift;
      need -= above;
    }
    // output row staged in the (now free) histogram when it fits
    int32_t* ostage = p.k <= 2048 ? reinterpret_cast<int32_t*>(sm->hist) : out;
    select_staged(keys4, nq, mask, prefix, need, ostage, p.k, sm);
    if (ostage != out) {
      __syncthreads();
      for (int j = tid; j < p.k; j += kThreads) out[j] = ostage[j];
    }
    if (p.count && tid == 0) p.count[row] = p.k;
    return;
  }
  // ---- rows longer than the shared stage: 4 x 8-bit passes re-reading the row (L2)
  auto key_at = [&](int s) -> uint32_t {
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
  p.stage_cap = (p.stage_cap + 3) & ~3;   // whole uint4 groups
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
