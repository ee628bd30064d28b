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
//            there (16-byte asynchronous copies). The first level bins key >> 17
//            (64 bins per octave) over 32 octaves of the sign where a 512-score
//            sample puts the k-th largest score, with one bin each for the keys
//            below and above that window; it is built while the keys are
//            converted. When at most kCandCap keys share the threshold bin, one
//            sweep writes the bitmap of the keys above it and the list of the keys
//            in it; the remaining digits are resolved on the list, whose selected
//            keys join the bitmaps, and one bitmap word per thread emits the
//            selection in ascending order (through a shared staging row for
//            coalesced stores). Otherwise 11 + 11 + 10 bit levels run over all
//            staged keys and an ordered sweep per warp segment writes the result.
//            Longer rows take 4 x 8-bit passes over global memory (L2) with
//            warp-aggregated (__match_any_sync) histograms. Every selection takes
//            the keys > T and the lowest-index `need` keys == T. Slots m..k-1
//            get -1.

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kStageMax = 16384;   // keys staged in shared memory per row
constexpr int kCandCap = 1024;     // threshold-bin keys resolved as a list
static_assert(kStageMax <= 32 * kThreads, "one bitmap word per thread");

struct TopkParams {
  const float* scores;
  long long ld;
  const int32_t* seg;
  int B, S, k;
  int32_t* idx;
  int32_t* count;
  int stage_cap;
  int t_lo, t_hi;        // the query rows of this launch (all of them, or one block)
  long long rows_blk;    // rows per batch of the score buffer: row t is its row t - t_lo
};

// the scores of query row t of batch row b
__device__ __forceinline__ const float* score_row(const TopkParams& p, int b, int t) {
  return p.scores + (static_cast<long long>(b) * p.rows_blk + (t - p.t_lo)) * p.ld;
}

struct TopkSmem {
  uint32_t hist[2048];
  int warp_tot[kWarps];
  int wgt[kWarps], weq[kWarps];
  int bcast[4];
  uint32_t ubc[4];
};

// Larger float -> larger key; -0.0 and +0.0 map to the same key; key 0 is never
// produced by a non-NaN score and marks an invalid (masked) key.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  // negative: all bits flipped; otherwise the sign bit set
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
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
  // up to 4 bins per thread (nb <= 4 * kThreads), the highest bins to thread 0
  const int per = nb > kThreads ? nb / kThreads : 1;
  const int tid = threadIdx.x;
  int c[4] = {0, 0, 0, 0};
  int sum = 0;
  for (int i = 0; i < per; ++i) {
    const int j = tid * per + i;
    c[i] = j < nb ? static_cast<int>(hist[nb - 1 - j]) : 0;
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

// First-level bins: h = key >> 17 (sign, exponent and six mantissa bits) over a
// window of 2046 values of h (32 octaves of one sign); bin 0 takes the keys below
// the window and bin 2047 the keys above it. The keys of a window bin share one
// 15-bit prefix.
struct LevelOne {
  uint32_t base;   // h of bin 1
  __device__ __forceinline__ uint32_t bucket(uint32_t key) const {
    const uint32_t h = key >> 17;
    return h < base ? 0u : min(h - base + 1u, 2047u);
  }
  __device__ __forceinline__ bool interior(uint32_t bin) const {
    return bin >= 1u && bin <= 2046u;
  }
  __device__ __forceinline__ uint32_t prefix(uint32_t bin) const {
    return (base + bin - 1u) << 17;
  }
  // From the largest positive score bits, the largest negative-score magnitude
  // bits and whether the k-th largest score is expected to be >= 0: the window
  // ends two octaves above the positive maximum, or starts two octaves beyond the
  // negative one.
  static __device__ __forceinline__ LevelOne make(uint32_t apos, uint32_t aneg,
                                                  bool positive_side) {
    LevelOne w;
    if (positive_side) {
      const uint32_t whi = min(0x4000u + (apos >> 17) + 128u, 0x7FFFu);
      w.base = whi - 2045u;
    } else {
      const uint32_t ha = (0x7FFFFFFFu - aneg) >> 17;
      w.base = ha > 128u ? ha - 128u : 0u;
    }
    return w;
  }
};

// Selection when the first level leaves at most kCandCap keys in the threshold bin
// ((key & 0xFFFE0000) == prefix): one sweep over the staged keys writes the
// bitmap of the keys above the bin and the list of the keys in it; the remaining
// digits are resolved on that list alone; the selected list keys are added to the
// bitmaps (above T / equal to T) and one word per thread emits the selection in
// ascending order, the first `need` keys equal to T included. The histogram area
// holds the bitmaps, the list and the small histogram, and then the output row.
__device__ __forceinline__ void select_candidates(const uint32_t* keys, const uint4* keys4,
                                                  int len, int nq, const LevelOne& w1,
                                                  uint32_t bin1, int need, int in_bin,
                                                  int32_t* out, int kmax, TopkSmem* sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t* gtw = sm->hist;                                     // [512] above T
  uint32_t* eqw = sm->hist + 512;                               // [512] equal to T
  uint16_t* cand = reinterpret_cast<uint16_t*>(sm->hist + 1024);   // [kCandCap]
  uint32_t* h2 = sm->hist + 1536;                               // [512]
  const bool inner = w1.interior(bin1);
  uint32_t mask = inner ? 0xFFFE0000u : 0u;
  uint32_t prefix = inner ? w1.prefix(bin1) : 0u;
  const int nwords = (len + 31) >> 5;
  const int ncand = in_bin;
  for (int i = tid; i < 512; i += kThreads) eqw[i] = 0u;
  if (tid == 0) sm->ubc[3] = 0u;
  __syncthreads();
  const uint32_t lt = (1u << lane) - 1u;
  for (int c0 = 0; c0 < nq; c0 += kThreads) {
    const int c = c0 + tid;
    uint32_t kk[4] = {0u, 0u, 0u, 0u};
    if (c < nq) {
      const uint4 kv = keys4[c];
      kk[0] = kv.x;
      kk[1] = kv.y;
      kk[2] = kv.z;
      kk[3] = kv.w;
    }
    uint32_t nib = 0u;
    bool cd[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t b1 = w1.bucket(kk[e]);
      nib |= static_cast<uint32_t>(kk[e] != 0u && b1 > bin1) << e;
      cd[e] = kk[e] != 0u && b1 == bin1;
    }
    // lanes 8j..8j+7 hold the 32 keys of one bitmap word
    uint32_t wv = nib << (4 * (lane & 7));
    wv |= __shfl_xor_sync(0xffffffffu, wv, 1);
    wv |= __shfl_xor_sync(0xffffffffu, wv, 2);
    wv |= __shfl_xor_sync(0xffffffffu, wv, 4);
    if ((lane & 7) == 0 && c < nq) gtw[c >> 3] = wv;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t bal = __ballot_sync(0xffffffffu, cd[e]);
      if (bal) {
        const int leader = __ffs(bal) - 1;
        uint32_t base = 0u;
        if (lane == leader) base = atomicAdd(&sm->ubc[3], static_cast<uint32_t>(__popc(bal)));
        base = __shfl_sync(0xffffffffu, base, leader);
        const uint32_t r = base + __popc(bal & lt);
        if (cd[e] && r < kCandCap) cand[r] = static_cast<uint16_t>(4 * c + e);
      }
    }
  }
  __syncthreads();
  // remaining digits on the list: bits 16..8 and 7..0 of an interior bin,
  // four bytes otherwise
  const int nlev = inner ? 2 : 4;
  int cur = in_bin;
#pragma unroll 1
  for (int lvl = 0; lvl < nlev && cur != need; ++lvl) {
    const int shift = inner ? 8 - 8 * lvl : 24 - 8 * lvl;
    const int nb = inner && lvl == 0 ? 512 : 256;
    const uint32_t low = (1u << shift) - 1u;
    for (int i = tid; i < nb; i += kThreads) h2[i] = 0u;
    if (tid == 0) {
      sm->ubc[1] = 0u;
      sm->ubc[2] = 0xFFFFFFFFu;
    }
    __syncthreads();
    uint32_t lo_or = 0u, lo_and = 0xFFFFFFFFu;
    for (int j = tid; j < ncand; j += kThreads) {
      const uint32_t key = keys[cand[j]];
      if ((key & mask) == prefix) {
        atomicAdd(&h2[(key >> shift) & static_cast<uint32_t>(nb - 1)], 1u);
        lo_or |= key & low;
        lo_and &= key & low;
      }
    }
    lo_or = __reduce_or_sync(0xffffffffu, lo_or);
    lo_and = __reduce_and_sync(0xffffffffu, lo_and);
    if (lane == 0) {
      atomicOr(&sm->ubc[1], lo_or);
      atomicAnd(&sm->ubc[2], lo_and);
    }
    __syncthreads();
    const uint32_t all_or = sm->ubc[1], all_and = sm->ubc[2];
    int bin, above;
    find_bin(h2, nb, need, sm, bin, above, cur);
    prefix |= static_cast<uint32_t>(bin) << shift;
    mask |= static_cast<uint32_t>(nb - 1) << shift;
    need -= above;
    if (all_or == (all_and & low)) {
      prefix |= all_or;
      mask |= low;
      break;
    }
  }
  // list keys above T / equal to T into the bitmaps
  for (int j = tid; j < ncand; j += kThreads) {
    const int sj = cand[j];
    const uint32_t km = keys[sj] & mask;
    if (km > prefix) atomicOr(&gtw[sj >> 5], 1u << (sj & 31));
    else if (km == prefix) atomicOr(&eqw[sj >> 5], 1u << (sj & 31));
  }
  __syncthreads();
  // one word per thread: offsets by a block scan of (above count | equal count << 16)
  uint32_t g = 0u, q = 0u;
  if (tid < nwords) {
    g = gtw[tid];
    q = eqw[tid];
  }
  const int own = __popc(g) | (__popc(q) << 16);
  int tot;
  const int excl = block_scan(own, tot, sm) - own;   // every word is read before this returns
  int gb = excl & 0xFFFF, eb = excl >> 16;
  int32_t* ost = kmax <= 2048 ? reinterpret_cast<int32_t*>(sm->hist) : out;
  uint32_t bits = g | q;
  while (bits) {
    const int b = __ffs(bits) - 1;
    bits &= bits - 1u;
    const int sj = tid * 32 + b;
    if ((g >> b) & 1u) {
      const int pos = gb + min(eb, need);
      if (pos < kmax) ost[pos] = sj;
      ++gb;
    } else {
      if (eb < need && gb + eb < kmax) ost[gb + eb] = sj;
      ++eb;
    }
  }
  if (ost != out) {
    __syncthreads();
    for (int j = tid; j < kmax; j += kThreads) out[j] = ost[j];
  }
}

__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkSmem* sm = reinterpret_cast<TopkSmem*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + sizeof(TopkSmem));

  // rows t_lo <= t < min(t_hi, stage_cap) of every batch row, long rows first
  const int sc = min(p.t_hi, p.stage_cap) - p.t_lo;
  const long long i = static_cast<long long>(gridDim.x) - 1 - blockIdx.x;
  const int b = static_cast<int>(i / sc);
  const int t = p.t_lo + static_cast<int>(i - static_cast<long long>(b) * sc);
  const long long row = static_cast<long long>(b) * p.S + t;
  const int len = t + 1;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int32_t* seg_row = p.seg ? p.seg + static_cast<long long>(b) * p.S : nullptr;
  const int seg_t = seg_row ? seg_row[t] : 0;
  const float* srow = score_row(p, b, t);
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

  {
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
    if (tid == 0) {
      sm->ubc[0] = 0u;
      sm->ubc[1] = 0u;
      sm->ubc[2] = 0u;
      sm->ubc[3] = 0u;
    }
    cp_async_wait<0>();
    __syncthreads();
    const int nq = (len + 3) >> 2;
    uint4* keys4 = reinterpret_cast<uint4*>(keys);
    // first-level window from up to 512 evenly spread valid scores (from the
    // whole row when none of them is valid): the largest positive score, the
    // largest negative magnitude and the share of scores >= 0
    uint32_t npos, nval;
    {
      const int si = static_cast<int>((static_cast<long long>(tid) * len) / kThreads);
      const bool v = !seg_row || seg_row[si] == seg_t;
      const uint32_t u = keys[si];
      const bool pos = v && ((u & 0x80000000u) == 0u || u == 0x80000000u);
      const uint32_t ap = __reduce_max_sync(0xffffffffu, pos ? (u & 0x7FFFFFFFu) : 0u);
      const uint32_t an = __reduce_max_sync(0xffffffffu, v && !pos ? (u & 0x7FFFFFFFu) : 0u);
      if (lane == 0) {
        atomicMax(&sm->ubc[0], ap);
        atomicMax(&sm->ubc[1], an);
      }
      npos = static_cast<uint32_t>(__syncthreads_count(pos));
      nval = static_cast<uint32_t>(__syncthreads_count(v));
    }
    if (nval == 0u) {
      uint32_t ap = 0u, an = 0u, cp = 0u, cv = 0u;
      for (int si = tid; si < len; si += kThreads) {
        if (seg_row[si] != seg_t) continue;
        const uint32_t u = keys[si];
        const bool pos = (u & 0x80000000u) == 0u || u == 0x80000000u;
        if (pos) ap = max(ap, u & 0x7FFFFFFFu);
        else an = max(an, u & 0x7FFFFFFFu);
        cp += pos;
        ++cv;
      }
      ap = __reduce_max_sync(0xffffffffu, ap);
      an = __reduce_max_sync(0xffffffffu, an);
      cp = __reduce_add_sync(0xffffffffu, cp);
      cv = __reduce_add_sync(0xffffffffu, cv);
      if (lane == 0) {
        atomicMax(&sm->ubc[0], ap);
        atomicMax(&sm->ubc[1], an);
        atomicAdd(&sm->ubc[2], cp);
        atomicAdd(&sm->ubc[3], cv);
      }
      __syncthreads();
      npos = sm->ubc[2];
      nval = sm->ubc[3];
    }
    // the k-th largest score is expected >= 0 when at least k of the n valid
    // scores are expected >= 0
    const bool positive_side =
        static_cast<unsigned long long>(npos) * n >= static_cast<unsigned long long>(nval) * p.k;
    const LevelOne w1 = LevelOne::make(sm->ubc[0], sm->ubc[1], positive_side);
    // order keys in place (invalid -> 0; the tail of the last uint4 -> 0) and the
    // first-level histogram, four consecutive keys per thread
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
        if (kq[e] != 0u) atomicAdd(&sm->hist[w1.bucket(kq[e])], 1u);
    }
    __syncthreads();
    int bin, above, in_bin;
    find_bin(sm->hist, 2048, p.k, sm, bin, above, in_bin);
    if (in_bin <= kCandCap) {
      select_candidates(keys, keys4, len, nq, w1, static_cast<uint32_t>(bin), p.k - above,
                        in_bin, out, p.k, sm);
      if (p.count && tid == 0) p.count[row] = p.k;
      return;
    }
    // many keys share the threshold bin: 11 + 11 + 10 bit levels over all staged
    // keys
    uint32_t prefix = 0u, mask = 0u;
    int need = p.k;
    in_bin = -1;
    const int shifts[3] = {21, 10, 0};
    const int nbins[3] = {2048, 2048, 1024};
    const int nlev = 3;
#pragma unroll 1
    for (int lvl = 0; lvl < nlev && in_bin != need; ++lvl) {
      const int shift = shifts[lvl], nb = nbins[lvl];
      const uint32_t low = (1u << shift) - 1u;
      for (int i = tid; i < nb; i += kThreads) sm->hist[i] = 0u;
      if (tid == 0) {
        sm->ubc[1] = 0u;            // OR of the bits below this level
        sm->ubc[2] = 0xFFFFFFFFu;   // AND of the bits below this level
      }
      __syncthreads();
      uint32_t lo_or = 0u, lo_and = 0xFFFFFFFFu;
      for (int c = tid; c < nq; c += kThreads) {
        const uint4 kv = keys4[c];
        const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (kk[e] != 0u && (kk[e] & mask) == prefix) {
            atomicAdd(&sm->hist[(kk[e] >> shift) & static_cast<uint32_t>(nb - 1)], 1u);
            lo_or |= kk[e] & low;
            lo_and &= kk[e] & low;
          }
      }
      lo_or = __reduce_or_sync(0xffffffffu, lo_or);
      lo_and = __reduce_and_sync(0xffffffffu, lo_and);
      if (lane == 0) {
        atomicOr(&sm->ubc[1], lo_or);
        atomicAnd(&sm->ubc[2], lo_and);
      }
      __syncthreads();
      const uint32_t all_or = sm->ubc[1], all_and = sm->ubc[2];
      find_bin(sm->hist, nb, need, sm, bin, above, in_bin);
      prefix |= static_cast<uint32_t>(bin) << shift;
      mask |= static_cast<uint32_t>(nb - 1) << shift;
      need -= above;
      if (all_or == (all_and & low)) {
        // every key still in play has the same lower bits: the key is resolved
        prefix |= all_or;
        mask |= low;
        break;
      }
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
  // rows longer than the shared stage are handled by topk_long_kernel
}

// ------------------------------------------------------------------ long rows
// Rows longer than the shared stage (t >= kStageMax): one persistent CTA of 1024
// threads per SM, so that the rows in flight (152 x at most 512 KB at S = 131072)
// stay in L2 between passes. Every pass reads the row from global memory in
// 16-byte groups of four keys: the first from DRAM (first-level histogram), the
// following ones from L2. The selection is the same as for staged rows: a window
// histogram, then either a candidate list with bitmaps (rows of at most
// kLongWords * 32 keys and at most kLongCand keys in the threshold bin) or further
// levels over the row with an ordered sweep.
namespace lr {

constexpr int NT = 1024;
constexpr int NW = NT / 32;
constexpr int kLongWords = 4096;   // bitmap words: rows up to 131072 keys
// candidates of the one-pass path: each warp appends to its own segment of 256; at
// S = 131072 a row leaves about 3.3K candidates, ~105 per warp, and segments of 128
// overflowed on about half of the rows beyond t = 90K
constexpr int kLongCand = 8192;
constexpr int kWpt = kLongWords / NT;   // bitmap words per thread

struct Smem {
  uint32_t hist[2048];
  uint32_t gtw[kLongWords];   // keys above T
  uint32_t eqw[kLongWords];   // keys equal to T
  uint32_t cand[kLongCand];   // threshold-bin key indices; then the output row
  int warp_tot[NW];
  int wgt[NW], weq[NW];
  int bcast[4];
  uint32_t ubc[8];
  int wcnt[NW];               // one-pass path: candidates appended by each warp
  uint32_t ckey[kLongCand];   // one-pass path: the order key of each candidate
};

// keys of one row read from global memory (tail of the last group and other
// documents' keys read as 0; the row stride is a multiple of 4 and at least S)
struct RowKeys {
  const float* srow;
  const int32_t* seg_row;
  int len, seg_t;
  __device__ __forceinline__ uint4 load4(int c) const {
    const float4 f = __ldg(reinterpret_cast<const float4*>(srow) + c);
    const float fv[4] = {f.x, f.y, f.z, f.w};
    uint32_t kq[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int si = 4 * c + e;
      const bool v = si < len && (!seg_row || __ldg(seg_row + si) == seg_t);
      kq[e] = v ? order_key(fv[e]) : 0u;
    }
    return make_uint4(kq[0], kq[1], kq[2], kq[3]);
  }
  // a group of four keys of the row with no segment ids (4c + 3 < len)
  __device__ __forceinline__ uint4 load4_full(int c) const {
    const float4 f = __ldg(reinterpret_cast<const float4*>(srow) + c);
    return make_uint4(order_key(f.x), order_key(f.y), order_key(f.z), order_key(f.w));
  }
  __device__ __forceinline__ uint32_t key(int s) const { return order_key(__ldg(srow + s)); }
};

__device__ __forceinline__ int block_scan(int v, int& total, Smem* sm) {
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
    int w = lane < NW ? sm->warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NW) sm->warp_tot[lane] = w;
  }
  __syncthreads();
  const int before = warp > 0 ? sm->warp_tot[warp - 1] : 0;
  total = sm->warp_tot[NW - 1];
  __syncthreads();
  return x + before;
}

// the bin of the need-th largest key among nb bins (nb <= 2 * NT), keys above it
// and in it
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nb, int need, Smem* sm,
                                         int& bin, int& above, int& in_bin) {
  const int per = nb > NT ? nb / NT : 1;
  const int tid = threadIdx.x;
  int c[2];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int j = tid * per + i;
    c[i] = i < per && j < nb ? static_cast<int>(hist[nb - 1 - j]) : 0;
    sum += c[i];
  }
  int tot;
  const int incl = block_scan(sum, tot, sm);
  int run = incl - sum;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (i < per && run < need && run + c[i] >= need) {
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

// digits below a known prefix over the keys visit(fn) presents (see the staged
// path: histogram levels, early stop when the bin holds exactly the keys needed
// or every key in play has the same lower bits)
template <class Visit>
__device__ __forceinline__ void resolve_levels(Visit visit, uint32_t* hist, int nlev,
                                               const int* shifts, const int* nbins,
                                               uint32_t& prefix, uint32_t& mask, int& need,
                                               int in_bin, Smem* sm) {
  const int tid = threadIdx.x, lane = tid & 31;
#pragma unroll 1
  for (int lvl = 0; lvl < nlev && in_bin != need; ++lvl) {
    const int shift = shifts[lvl], nb = nbins[lvl];
    const uint32_t low = (1u << shift) - 1u;
    for (int i = tid; i < nb; i += NT) hist[i] = 0u;
    if (tid == 0) {
      sm->ubc[4] = 0u;
      sm->ubc[5] = 0xFFFFFFFFu;
    }
    __syncthreads();
    uint32_t lo_or = 0u, lo_and = 0xFFFFFFFFu;
    const uint32_t pf = prefix, mk = mask;
    visit([&](uint32_t key) {
      if (key != 0u && (key & mk) == pf) {
        atomicAdd(&hist[(key >> shift) & static_cast<uint32_t>(nb - 1)], 1u);
        lo_or |= key & low;
        lo_and &= key & low;
      }
    });
    lo_or = __reduce_or_sync(0xffffffffu, lo_or);
    lo_and = __reduce_and_sync(0xffffffffu, lo_and);
    if (lane == 0) {
      atomicOr(&sm->ubc[4], lo_or);
      atomicAnd(&sm->ubc[5], lo_and);
    }
    __syncthreads();
    const uint32_t all_or = sm->ubc[4], all_and = sm->ubc[5];
    int bin, above;
    find_bin(hist, nb, need, sm, bin, above, in_bin);
    prefix |= static_cast<uint32_t>(bin) << shift;
    mask |= static_cast<uint32_t>(nb - 1) << shift;
    need -= above;
    if (all_or == (all_and & low)) {
      prefix |= all_or;
      mask |= low;
      break;
    }
  }
}

// ordered selection over the row by per-warp segments (count sweep, write sweep)
__device__ __forceinline__ void select_sweep(const RowKeys& rk, int nq, uint32_t mask,
                                             uint32_t prefix, int need, int32_t* out, int kmax,
                                             Smem* sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int segq = ((nq + NW * 32 - 1) / (NW * 32)) * 32;
  const int q_begin = warp * segq, q_end = min(nq, q_begin + segq);
  int cg = 0, ce = 0;
  for (int q = q_begin + lane; q < q_end; q += 32) {
    const uint4 kv = rk.load4(q);
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
      const uint4 kv = rk.load4(q);
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
  __syncthreads();   // wgt / weq are reused by the next row
}

// The selection from the candidate list sm->cand[0..in_bin) (every key that can still
// be selected beyond those already marked in sm->gtw): the remaining digits below
// (prefix, mask), the candidates marked above / equal to the threshold, and the
// ascending emission of the gtw keys and the first `need` eqw keys.
__device__ __forceinline__ void finish_candidates(const RowKeys& rk, bool inner, uint32_t prefix,
                                                  uint32_t mask, int need, int in_bin, int nwords,
                                                  const TopkParams& p, int32_t* out, Smem* sm) {
  const int tid = threadIdx.x;
  const int ncand = min(in_bin, kLongCand);
  const int shifts_in[2] = {8, 0}, nbins_in[2] = {512, 256};
  const int shifts_out[4] = {24, 16, 8, 0}, nbins_out[4] = {256, 256, 256, 256};
  resolve_levels(
      [&](auto fn) {
        for (int j = tid; j < ncand; j += NT) fn(rk.key(static_cast<int>(sm->cand[j])));
      },
      sm->hist, inner ? 2 : 4, inner ? shifts_in : shifts_out, inner ? nbins_in : nbins_out,
      prefix, mask, need, in_bin, sm);
  for (int j = tid; j < ncand; j += NT) {
    const int sj = static_cast<int>(sm->cand[j]);
    const uint32_t km = rk.key(sj) & mask;
    if (km > prefix) atomicOr(&sm->gtw[sj >> 5], 1u << (sj & 31));
    else if (km == prefix) atomicOr(&sm->eqw[sj >> 5], 1u << (sj & 31));
  }
  __syncthreads();
  uint32_t g[kWpt], q[kWpt];
  int own = 0;
#pragma unroll
  for (int i = 0; i < kWpt; ++i) {
    const int wd = tid * kWpt + i;
    g[i] = wd < nwords ? sm->gtw[wd] : 0u;
    q[i] = wd < nwords ? sm->eqw[wd] : 0u;
    own += __popc(g[i]) | (__popc(q[i]) << 16);
  }
  int tot;
  const int excl = block_scan(own, tot, sm) - own;   // every word is read before this returns
  int gb = excl & 0xFFFF, eb = excl >> 16;
  int32_t* ost = p.k <= kLongCand ? reinterpret_cast<int32_t*>(sm->cand) : out;
#pragma unroll
  for (int i = 0; i < kWpt; ++i) {
    uint32_t bits = g[i] | q[i];
    while (bits) {
      const int bb = __ffs(bits) - 1;
      bits &= bits - 1u;
      const int sj = (tid * kWpt + i) * 32 + bb;
      if ((g[i] >> bb) & 1u) {
        const int pos = gb + min(eb, need);
        if (pos < p.k) ost[pos] = sj;
        ++gb;
      } else {
        if (eb < need && gb + eb < p.k) ost[gb + eb] = sj;
        ++eb;
      }
    }
  }
  __syncthreads();
  if (ost != out)
    for (int j = tid; j < p.k; j += NT) out[j] = ost[j];
}

__device__ __forceinline__ void select_row(const RowKeys& rk, int t, int n, const TopkParams& p,
                                           int32_t* out, long long row, Smem* sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int len = t + 1;
  const int nq = (len + 3) >> 2;
  if (n <= p.k) {
    // every valid key is selected: an ordered sweep taking every valid key as
    // "equal" (mask 0) with need = k >= n
    select_sweep(rk, nq, 0u, 0u, p.k, out, p.k, sm);
    for (int j = n + tid; j < p.k; j += NT) out[j] = -1;
    if (p.count && tid == 0) p.count[row] = n;
    return;
  }
  // ---- one pass: every key at or above a threshold placed from a strided sample (one
  // group of 4 keys per thread, evenly spaced over the row) at the sample rank that k
  // takes in the row plus four standard deviations. When that leaves between k and
  // kLongCand keys, the top k are among them and the candidate finish selects them
  // exactly; otherwise the two-pass path below runs.
  const int nwords0 = (4 * nq + 31) >> 5;
  if (nwords0 <= kLongWords) {
    for (int i = tid; i < 2048; i += NT) sm->hist[i] = 0u;
    if (tid < 8) sm->ubc[tid] = 0u;
    const int cs = static_cast<int>((static_cast<long long>(tid) * nq) / NT);
    const uint4 smp = rk.load4(cs);
    const uint32_t sk[4] = {smp.x, smp.y, smp.z, smp.w};
    uint32_t ap = 0u, an = 0u, cp = 0u, cv = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (sk[e] == 0u) continue;
      const bool pos = sk[e] >= 0x80000000u;
      if (pos) ap = max(ap, sk[e] & 0x7FFFFFFFu);
      else an = max(an, ~sk[e] & 0x7FFFFFFFu);
      cp += pos;
      ++cv;
    }
    ap = __reduce_max_sync(0xffffffffu, ap);
    an = __reduce_max_sync(0xffffffffu, an);
    cp = __reduce_add_sync(0xffffffffu, cp);
    cv = __reduce_add_sync(0xffffffffu, cv);
    __syncthreads();
    if (lane == 0) {
      atomicMax(&sm->ubc[0], ap);
      atomicMax(&sm->ubc[1], an);
      atomicAdd(&sm->ubc[2], cp);
      atomicAdd(&sm->ubc[3], cv);
    }
    __syncthreads();
    const uint32_t npos = sm->ubc[2], nval = sm->ubc[3];
    if (nval > 0u) {
      const bool positive_side = static_cast<unsigned long long>(npos) * n >=
                                 static_cast<unsigned long long>(nval) * p.k;
      const LevelOne ws = LevelOne::make(sm->ubc[0], sm->ubc[1], positive_side);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (sk[e] != 0u) atomicAdd(&sm->hist[ws.bucket(sk[e])], 1u);
      __syncthreads();
      const float mu = static_cast<float>(p.k) * static_cast<float>(nval) / static_cast<float>(n);
      int rs = static_cast<int>(mu + 4.f * sqrtf(mu) + 8.f);
      if (rs > static_cast<int>(nval)) rs = static_cast<int>(nval);
      int sbin, sabove, sin_bin;
      find_bin(sm->hist, 2048, rs, sm, sbin, sabove, sin_bin);
      if (ws.interior(static_cast<uint32_t>(sbin))) {
        const uint32_t L = ws.prefix(static_cast<uint32_t>(sbin));
        for (int i = tid; i < nwords0; i += NT) {
          sm->gtw[i] = 0u;
          sm->eqw[i] = 0u;
        }
        for (int i = tid; i < 2048; i += NT) sm->hist[i] = 0u;   // now: the candidates' bins
        if (tid == 0) {
          sm->ubc[6] = 0u;
          sm->ubc[7] = 0u;
        }
        __syncthreads();
        // each warp appends to its own segment of the list, so that no counter is
        // shared between warps; a warp that fills its segment sends the row to the
        // two-pass path
        constexpr int kSeg = kLongCand / NW;
        const int wid = tid >> 5;
        uint32_t* seg = sm->cand + wid * kSeg;
        uint32_t* segk = sm->ckey + wid * kSeg;
        int wc = 0;
        const uint32_t lt = (1u << lane) - 1u;
        // invalid keys map to 0, every valid one to at least 1
        const uint32_t Lv = L > 0u ? L : 1u;
        // groups that lie wholly inside the row need no per-key validity when there are
        // no segment ids
        const int nfull = rk.seg_row ? 0 : len >> 2;
        for (int c0 = 0; c0 < nq; c0 += 4 * NT) {
          uint4 kv[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = c0 + u * NT + tid;
            kv[u] = c < nfull ? rk.load4_full(c)
                              : (c < nq ? rk.load4(c) : make_uint4(0u, 0u, 0u, 0u));
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint32_t kk[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
            const int c = c0 + u * NT + tid;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const bool cd = kk[e] >= Lv;
              const uint32_t bal = __ballot_sync(0xffffffffu, cd);
              const int r = wc + __popc(bal & lt);
              if (cd && r < kSeg) {
                seg[r] = static_cast<uint32_t>(4 * c + e);
                segk[r] = kk[e];
              }
              wc += __popc(bal);
            }
          }
        }
        if (lane == 0) {
          sm->wcnt[wid] = wc;
          if (wc > kSeg) sm->ubc[6] = 1u;   // a segment overflowed
          atomicAdd(&sm->ubc[7], static_cast<uint32_t>(wc));
        }
        // the candidates' first-level bins, after the pass (a few thousand keys)
        for (int j = lane; j < min(wc, kSeg); j += 32) atomicAdd(&sm->hist[ws.bucket(segk[j])], 1u);
        __syncthreads();
        const int C = static_cast<int>(sm->ubc[7]);
        const bool fits = sm->ubc[6] == 0u;
        __syncthreads();
        if (tid == 0) sm->ubc[7] = 0u;   // reused as the in-bin counter below
        __syncthreads();
        int bin = 0, above = 0, in_bin = 0;
        // every key >= L is a candidate and there are at least k: the bin of the k-th
        // largest candidate is the row's threshold bin
        if (fits && C >= p.k) find_bin(sm->hist, 2048, p.k, sm, bin, above, in_bin);
        if (fits && C >= p.k && in_bin <= kLongWords) {
          // candidates above the threshold bin go to the bitmap, those in it become the
          // list (staged in eqw, which is zeroed after)
          const uint32_t b1 = static_cast<uint32_t>(bin);
          for (int j = lane; j < sm->wcnt[wid]; j += 32) {
            const uint32_t sj = seg[j];
            const uint32_t bk = ws.bucket(segk[j]);
            if (bk > b1) {
              atomicOr(&sm->gtw[sj >> 5], 1u << (sj & 31));
            } else if (bk == b1) {
              const uint32_t r = atomicAdd(&sm->ubc[7], 1u);
              sm->eqw[r] = sj;
            }
          }
          __syncthreads();
          for (int j = tid; j < in_bin; j += NT) sm->cand[j] = sm->eqw[j];
          __syncthreads();
          for (int i = tid; i < nwords0; i += NT) sm->eqw[i] = 0u;
          __syncthreads();
          const bool inner = ws.interior(b1);
          finish_candidates(rk, inner, inner ? ws.prefix(b1) : 0u, inner ? 0xFFFE0000u : 0u,
                            p.k - above, in_bin, nwords0, p, out, sm);
          if (p.count && tid == 0) p.count[row] = p.k;
          __syncthreads();   // the shared state is reused by the next row
          return;
        }
        __syncthreads();   // C is read before the two-pass path resets the counters
      }
    }
  }
  for (int i = tid; i < 2048; i += NT) sm->hist[i] = 0u;
  if (tid < 4) sm->ubc[tid] = 0u;
  // the first group of each thread (the row's first 4096 keys) places the window
  const uint4 first = tid < nq ? rk.load4(tid) : make_uint4(0u, 0u, 0u, 0u);
  {
    const uint32_t fk[4] = {first.x, first.y, first.z, first.w};
    uint32_t ap = 0u, an = 0u, cp = 0u, cv = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (fk[e] == 0u) continue;
      const bool pos = fk[e] >= 0x80000000u;
      if (pos) ap = max(ap, fk[e] & 0x7FFFFFFFu);
      else an = max(an, ~fk[e] & 0x7FFFFFFFu);
      cp += pos;
      ++cv;
    }
    ap = __reduce_max_sync(0xffffffffu, ap);
    an = __reduce_max_sync(0xffffffffu, an);
    cp = __reduce_add_sync(0xffffffffu, cp);
    cv = __reduce_add_sync(0xffffffffu, cv);
    __syncthreads();
    if (lane == 0) {
      atomicMax(&sm->ubc[0], ap);
      atomicMax(&sm->ubc[1], an);
      atomicAdd(&sm->ubc[2], cp);
      atomicAdd(&sm->ubc[3], cv);
    }
    __syncthreads();
  }
  const uint32_t npos = sm->ubc[2], nval = sm->ubc[3];
  const bool positive_side = nval == 0u || static_cast<unsigned long long>(npos) * n >=
                                               static_cast<unsigned long long>(nval) * p.k;
  const LevelOne w1 = LevelOne::make(sm->ubc[0], sm->ubc[1], positive_side);
  // first-level histogram over the row (four groups in flight per thread)
  {
    int c = tid;
    if (c < nq) {
      const uint32_t kk[4] = {first.x, first.y, first.z, first.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (kk[e] != 0u) atomicAdd(&sm->hist[w1.bucket(kk[e])], 1u);
    }
    for (c += NT; c < nq; c += 4 * NT) {
      uint4 kv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        kv[u] = c + u * NT < nq ? rk.load4(c + u * NT) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t kk[4] = {kv[u].x, kv[u].y, kv[u].z, kv[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (kk[e] != 0u) atomicAdd(&sm->hist[w1.bucket(kk[e])], 1u);
      }
    }
  }
  __syncthreads();
  int bin, above, in_bin;
  find_bin(sm->hist, 2048, p.k, sm, bin, above, in_bin);
  const bool inner = w1.interior(static_cast<uint32_t>(bin));
  const int nwords = (4 * nq + 31) >> 5;
  if (nwords <= kLongWords && in_bin <= kLongCand) {
    // ---- candidate list and bitmaps
    uint32_t mask = inner ? 0xFFFE0000u : 0u;
    uint32_t prefix = inner ? w1.prefix(static_cast<uint32_t>(bin)) : 0u;
    int need = p.k - above;
    for (int i = tid; i < nwords; i += NT) sm->eqw[i] = 0u;
    if (tid == 0) sm->ubc[6] = 0u;
    __syncthreads();
    const uint32_t lt = (1u << lane) - 1u;
    const uint32_t b1 = static_cast<uint32_t>(bin);
    for (int c0 = 0; c0 < nq; c0 += NT) {
      const int c = c0 + tid;
      const uint4 kv = c < nq ? rk.load4(c) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t kk[4] = {kv.x, kv.y, kv.z, kv.w};
      uint32_t nib = 0u;
      bool cd[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t bk = w1.bucket(kk[e]);
        nib |= static_cast<uint32_t>(kk[e] != 0u && bk > b1) << e;
        cd[e] = kk[e] != 0u && bk == b1;
      }
      uint32_t wv = nib << (4 * (lane & 7));
      wv |= __shfl_xor_sync(0xffffffffu, wv, 1);
      wv |= __shfl_xor_sync(0xffffffffu, wv, 2);
      wv |= __shfl_xor_sync(0xffffffffu, wv, 4);
      if ((lane & 7) == 0 && c < nq) sm->gtw[c >> 3] = wv;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t bal = __ballot_sync(0xffffffffu, cd[e]);
        if (bal) {
          const int leader = __ffs(bal) - 1;
          uint32_t base = 0u;
          if (lane == leader) base = atomicAdd(&sm->ubc[6], static_cast<uint32_t>(__popc(bal)));
          base = __shfl_sync(0xffffffffu, base, leader);
          const uint32_t r = base + __popc(bal & lt);
          if (cd[e] && r < kLongCand) sm->cand[r] = static_cast<uint32_t>(4 * c + e);
        }
      }
    }
    __syncthreads();
    finish_candidates(rk, inner, prefix, mask, need, in_bin, nwords, p, out, sm);
  } else {
    // ---- further levels over the whole row
    uint32_t prefix = 0u, mask = 0u;
    int need = p.k;
    if (inner) {
      prefix = w1.prefix(static_cast<uint32_t>(bin));
      mask = 0xFFFE0000u;
      need = p.k - above;
    } else {
      in_bin = -1;
    }
    const int shifts_in[2] = {6, 0}, nbins_in[2] = {2048, 64};
    const int shifts_out[3] = {21, 10, 0}, nbins_out[3] = {2048, 2048, 1024};
    resolve_levels(
        [&](auto fn) {
          for (int c = tid; c < nq; c += NT) {
            const uint4 kv = rk.load4(c);
            fn(kv.x);
            fn(kv.y);
            fn(kv.z);
            fn(kv.w);
          }
        },
        sm->hist, inner ? 2 : 3, inner ? shifts_in : shifts_out, inner ? nbins_in : nbins_out,
        prefix, mask, need, in_bin, sm);
    select_sweep(rk, nq, mask, prefix, need, out, p.k, sm);
  }
  if (p.count && tid == 0) p.count[row] = p.k;
  __syncthreads();   // the shared state is reused by the next row
}

}  // namespace lr

// rows t0 <= t < t_hi of every batch row; persistent, longest rows first
__global__ void __launch_bounds__(lr::NT, 1) topk_long_kernel(const TopkParams p, int t0) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  lr::Smem* sm = reinterpret_cast<lr::Smem*>(smem_raw);
  const int tid = threadIdx.x;
  const long long nlong = static_cast<long long>(p.B) * (p.t_hi - t0);
  for (long long j = blockIdx.x; j < nlong; j += gridDim.x) {
    const int b = static_cast<int>(j % p.B);
    const int t = p.t_hi - 1 - static_cast<int>(j / p.B);
    const long long row = static_cast<long long>(b) * p.S + t;
    const int32_t* seg_row = p.seg ? p.seg + static_cast<long long>(b) * p.S : nullptr;
    const int seg_t = seg_row ? seg_row[t] : 0;
    int n = t + 1;
    if (seg_row) {
      int c = 0;
      for (int s = tid; s <= t; s += lr::NT) c += (seg_row[s] == seg_t);
      int tot;
      lr::block_scan(c, tot, sm);
      n = tot;
    }
    const lr::RowKeys rk{score_row(p, b, t), seg_row, t + 1, seg_t};
    lr::select_row(rk, t, n, p, p.idx + row * p.k, row, sm);
  }
}
}  // namespace

int launch_topk(const float* scores, int64_t ld, const int32_t* seg, int B, int S, int k,
                int32_t* idx, int32_t* count, cudaStream_t stream) {
  return launch_topk_rows(scores, ld, seg, B, S, k, idx, count, stream, 0, S, S);
}

int launch_topk_rows(const float* scores, int64_t ld, const int32_t* seg, int B, int S, int k,
                     int32_t* idx, int32_t* count, cudaStream_t stream, int t_lo, int t_hi,
                     long long rows_blk) {
  TopkParams p;
  p.scores = scores;
  p.ld = ld;
  p.seg = seg;
  p.B = B;
  p.S = S;
  p.k = k;
  p.idx = idx;
  p.count = count;
  p.t_lo = t_lo;
  p.t_hi = t_hi;
  p.rows_blk = rows_blk;
  p.stage_cap = S < kStageMax ? S : kStageMax;
  p.stage_cap = (p.stage_cap + 3) & ~3;   // whole uint4 groups
  const size_t smem = sizeof(TopkSmem) + static_cast<size_t>(p.stage_cap) * 4;
  if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  const long long rows = static_cast<long long>(B) * S;
  if (rows > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
  // rows t < stage_cap: one CTA per row with the row staged in shared memory
  const int short_hi = t_hi < p.stage_cap ? t_hi : p.stage_cap;
  if (short_hi > t_lo) {
    const long long nshort = static_cast<long long>(B) * (short_hi - t_lo);
    topk_kernel<<<static_cast<unsigned>(nshort), kThreads, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  }
  const int long_lo = t_lo > kStageMax ? t_lo : kStageMax;
  if (S > kStageMax && t_hi > long_lo) {
    // longer rows: persistent CTAs, one per SM
    const size_t lsmem = sizeof(lr::Smem);
    if (cudaFuncSetAttribute(topk_long_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(lsmem)) != cudaSuccess)
      return DSA_ERR_CUDA;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long nlong = static_cast<long long>(B) * (t_hi - long_lo);
    const int grid = static_cast<int>(nlong < sms ? nlong : sms);
    topk_long_kernel<<<grid, lr::NT, lsmem, stream>>>(p, long_lo);
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

}  // namespace dsa
