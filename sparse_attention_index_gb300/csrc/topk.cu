// Per-query top-k of the index scores: an exact block-wide radix select.
//
// ("DeepSeek3.2: Onboard sparse attention", Background: top-k token selection
// per query turns the index scores into the index mask. Equal scores go to the
// lower key index, -0.0 equals +0.0.)
//
// The valid keys of query row (b, t) are s in [0, t] with, when segment ids are
// given, seg[s] == seg[t]; n = their number. Scores are mapped to order-preserving
// 32-bit keys (-0 -> +0; 0 marks an invalid key).
//   n <= k : every valid key is selected (an ordered compaction).
//   n >  k : the k-th largest key T is found, and the keys > T and the lowest-index
//            `need` keys == T are emitted in ascending order from two bitmaps.
// Rows of at most kStageMax keys (sr::topk_short_kernel, one 256-thread CTA per row):
// a 2048-key sample places a window [L, U) around T; one sweep over the row sets the
// bitmap of the keys >= U and lists the keys in [L, U); T's digits are resolved on the
// list (a generic radix select over the row when the window misses). Longer rows
// (topk_long_kernel, one persistent 1024-thread CTA per SM) run the same selection with
// passes over the row in L2.
//
// Optionally each slot's score goes out too (vals, -inf at slots without a key): it is
// read back from the row while the row is still in L2, right after its selection, so
// that a consumer of the selected scores (the indexer loss) reads k contiguous floats
// per row instead of gathering them from the whole score row.

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kStageMax = 16384;   // rows of at most this many keys: the short-row kernel

struct TopkParams {
  const float* scores;
  long long ld;
  const int32_t* seg;
  int B, S, k;
  int32_t* idx;
  int32_t* count;
  float* vals;           // non-null: [B, S, k] scores of the selected keys, -inf past them
  int t_lo, t_hi;        // the query rows of this launch (all of them, or one block)
  long long rows_blk;    // rows per batch of the score buffer: row t is its row t - t_lo
  const int* gate;       // non-null: the launch does nothing unless *gate != 0
};

__device__ __forceinline__ bool gated_off(const TopkParams& p) {
  return p.gate != nullptr && *reinterpret_cast<const volatile int*>(p.gate) == 0;
}

// the scores of query row t of batch row b
__device__ __forceinline__ const float* score_row(const TopkParams& p, int b, int t) {
  return p.scores + (static_cast<long long>(b) * p.rows_blk + (t - p.t_lo)) * p.ld;
}

// Larger float -> larger key; -0.0 and +0.0 map to the same key; key 0 is never
// produced by a non-NaN score and marks an invalid (masked) key.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  // negative: all bits flipped; otherwise the sign bit set
  return u ^ (static_cast<uint32_t>(static_cast<int32_t>(u) >> 31) | 0x80000000u);
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

// ------------------------------------------------------------------ short rows
// Rows of at most kStageMax keys: one CTA of 256 threads per row, the row read from
// global memory (no staging), so that six or more rows are in flight per SM.
//   n <= k : an ordered compaction of the valid keys.
//   n >  k : a sample of 2048 keys (eight per thread, spread over the row) gives, by
//            its order statistics, two keys L < U with the k-th largest key T most
//            likely in [L, U): the sample rank of T, k * ns / n, plus / minus kZ
//            binomial standard deviations, placed by a coarse histogram of the sample
//            over the whole key range and a fine one inside the two coarse bins. One
//            coalesced sweep over the row sets the bitmap of the keys >= U, counts
//            them (A) and lists the keys in [L, U) with their indices. When
//            A <= k <= A + (listed keys) and the list fits, T lies in the list and
//            its remaining digits are resolved there; otherwise (a miss: rare) a
//            generic radix select over the row finds T. Either way the keys > T and
//            the lowest-index `need` keys == T are emitted in ascending order from
//            two bitmaps, through a shared staging row.
namespace sr {

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr int kWords = kStageMax / 32;   // bitmap words of the longest row
constexpr int kWpt = kWords / NT;        // bitmap words per thread
static_assert(kWpt == 2, "two bitmap words per thread");
constexpr int kCand = 2048;              // window keys held in shared memory
constexpr int kSampleGroups = 2;         // uint4 sample groups per thread
constexpr float kZ = 3.5f;               // window half-width in standard deviations
constexpr int kSweepDepth = 4;           // groups of four keys per thread in flight

struct Smem {
  uint32_t hist[2048];   // sample and level histograms, then the output row
  uint32_t gtw[kWords];  // keys above T
  uint32_t eqw[kWords];  // keys equal to T
  uint32_t cw[kWords];   // window keys (in [L, U))
  uint32_t ckey[kCand];  // window keys: the order key
  uint16_t cidx[kCand];  //   and the key index
  int warp_tot[NW];
  int bcast[4];
  uint32_t ubc[8];
};

template <class SM>
__device__ __forceinline__ int block_scan(int v, int& total, SM* sm) {
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
    for (int o = 1; o < NW; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < NW) sm->warp_tot[lane] = w;
  }
  __syncthreads();
  const int before = warp > 0 ? sm->warp_tot[warp - 1] : 0;
  total = sm->warp_tot[NW - 1];
  __syncthreads();   // warp_tot is reused by the next call
  return x + before;
}

// Over nb <= 2048 bins taken from the top: the bin holding the need-th largest key
// (need >= 1), the number of keys in higher bins and in that bin.
template <class SM>
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nb, int need, SM* sm,
                                         int& bin, int& above, int& in_bin) {
  const int per = nb > NT ? nb / NT : 1;
  const int tid = threadIdx.x;
  int c[8];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int j = tid * per + i;
    c[i] = i < per && j < nb ? static_cast<int>(hist[nb - 1 - j]) : 0;
    sum += c[i];
  }
  int tot;
  const int incl = block_scan(sum, tot, sm);
  int run = incl - sum;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
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

// the row's keys: order keys of the valid scores, 0 elsewhere (the row stride is a
// multiple of 4 and at least S, so every group of four inside the row can be read)
struct Row {
  const float* srow;
  const int32_t* seg_row;
  int len, seg_t;
  bool seg16;   // seg_row is 16-byte aligned: whole groups of four ids in one load
  // bit e: key 4c + e is valid
  __device__ __forceinline__ uint32_t valid4(int c) const {
    const int s0 = 4 * c;
    const uint32_t in_row = s0 + 3 < len ? 0xFu : (len > s0 ? (1u << (len - s0)) - 1u : 0u);
    if (!seg_row) return in_row;
    if (seg16 && s0 + 3 < len) {
      const int4 g = __ldg(reinterpret_cast<const int4*>(seg_row + s0));
      return static_cast<uint32_t>(g.x == seg_t) | static_cast<uint32_t>(g.y == seg_t) << 1 |
             static_cast<uint32_t>(g.z == seg_t) << 2 | static_cast<uint32_t>(g.w == seg_t) << 3;
    }
    uint32_t m = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (((in_row >> e) & 1u) && __ldg(seg_row + s0 + e) == seg_t) m |= 1u << e;
    return m;
  }
  // the raw scores of group c, NaN for the invalid keys
  __device__ __forceinline__ void load4f(int c, float (&f)[4]) const {
    const float4 v = __ldg(reinterpret_cast<const float4*>(srow) + c);
    f[0] = v.x;
    f[1] = v.y;
    f[2] = v.z;
    f[3] = v.w;
    if (seg_row || 4 * c + 3 >= len) {
      const uint32_t m = valid4(c);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (!((m >> e) & 1u)) f[e] = __int_as_float(0x7fc00000);
    }
  }
  __device__ __forceinline__ void load4(int c, uint32_t (&kq)[4]) const {
    const float4 f = __ldg(reinterpret_cast<const float4*>(srow) + c);
    const float fv[4] = {f.x, f.y, f.z, f.w};
    const uint32_t m = valid4(c);
#pragma unroll
    for (int e = 0; e < 4; ++e) kq[e] = ((m >> e) & 1u) ? order_key(fv[e]) : 0u;
  }
};

// lanes 8j..8j+7 of a warp hold the 32 keys of one bitmap word (four each): the word
__device__ __forceinline__ uint32_t gather_word(uint32_t nib, int lane) {
  uint32_t wv = nib << (4 * (lane & 7));
  wv |= __shfl_xor_sync(0xffffffffu, wv, 1);
  wv |= __shfl_xor_sync(0xffffffffu, wv, 2);
  wv |= __shfl_xor_sync(0xffffffffu, wv, 4);
  return wv;
}

// the keys > T (gtw) and the lowest-index `need` keys == T (eqw), `total` keys in all,
// into out[0, total) in ascending key index, and -1 into out[total, kmax); each thread
// owns words 2 * tid and 2 * tid + 1. With VALS, each slot's score from srow into vals as
// well (-inf past total).
template <bool VALS>
__device__ __forceinline__ void emit(int nwords, int need, int total, int32_t* out, int kmax,
                                     Smem* sm, const float* srow, float* vals) {
  const int tid = threadIdx.x;
  uint32_t g[kWpt], q[kWpt];
  int cg = 0, ce = 0;
#pragma unroll
  for (int i = 0; i < kWpt; ++i) {
    const int w = kWpt * tid + i;
    g[i] = w < nwords ? sm->gtw[w] : 0u;
    q[i] = w < nwords ? sm->eqw[w] : 0u;
    cg += __popc(g[i]);
    ce += __popc(q[i]);
  }
  const int own = cg | (ce << 16);
  int tot;
  const int excl = block_scan(own, tot, sm) - own;   // every word is read before this returns
  int eb = excl >> 16;
  // a selected key's slot = the selected keys before it: keys above T, and of the keys
  // equal to T the first `need` only
  int pos = (excl & 0xFFFF) + min(eb, need);
  int32_t* ost = kmax <= 2048 ? reinterpret_cast<int32_t*>(sm->hist) : out;
#pragma unroll
  for (int i = 0; i < kWpt; ++i) {
    uint32_t qk = 0u, m = q[i];
    for (int room = need - eb; m != 0u && room > 0; --room) {
      const uint32_t low = m & (0u - m);
      qk |= low;
      m ^= low;
    }
    eb += __popc(q[i]);
    uint32_t sel = g[i] | qk;
    while (sel) {
      const int bpos = __ffs(sel) - 1;
      sel &= sel - 1u;
      const int key = (kWpt * tid + i) * 32 + bpos;
      if (pos < kmax) {
        ost[pos] = key;
        if (VALS && ost == out) vals[pos] = __ldg(srow + key);
      }
      ++pos;
    }
  }
  if (ost != out) {
    __syncthreads();
    if (VALS) {
#pragma unroll 4
      for (int j = tid; j < kmax; j += NT) {
        const int key = j < total ? ost[j] : -1;
        out[j] = key;
        vals[j] = key >= 0 ? __ldg(srow + key) : -INFINITY;
      }
    } else {
      for (int j = tid; j < kmax; j += NT) out[j] = j < total ? ost[j] : -1;
    }
  } else {
    for (int j = total + tid; j < kmax; j += NT) {
      out[j] = -1;
      if (VALS) vals[j] = -INFINITY;
    }
  }
}

// a float x_t with  order_key(x) >= key  <=>  x >= x_t  for every non-NaN x: the float of
// that order key; NaN (nothing passes) above the key of +inf, -inf (everything passes) at
// or below the key of -inf
__device__ __forceinline__ float key_to_float(uint32_t key) {
  if (key > 0xFF800000u) return __int_as_float(0x7fc00000);
  if (key <= 0x007FFFFFu) return -INFINITY;
  return __uint_as_float(key >= 0x80000000u ? key ^ 0x80000000u : ~key);
}

// Remaining digits of T below the known bits `mask` (prefix) over the keys visit(fn)
// presents, in levels of up to max_bits (<= 11) bits from bit hb down: per level a
// histogram of the keys still in play, the bin of the need-th largest, and an early stop
// when that bin holds exactly the keys needed or every key in play has the same lower
// bits. A few hundred listed keys take 8-bit levels (one bin per thread to clear and
// scan); a whole row takes 11-bit ones.
template <class Visit, class SM>
__device__ __forceinline__ void resolve(Visit visit, int hb, uint32_t& prefix, uint32_t& mask,
                                        int& need, int cur, SM* sm, int max_bits = 11) {
  const int tid = threadIdx.x, lane = tid & 31;
#pragma unroll 1
  while (hb >= 0 && cur != need) {
    const int nbits = hb + 1 < max_bits ? hb + 1 : max_bits;
    const int shift = hb + 1 - nbits, nb = 1 << nbits;
    const uint32_t low = (1u << shift) - 1u;
    for (int i = tid; i < nb; i += NT) sm->hist[i] = 0u;
    if (tid == 0) {
      sm->ubc[4] = 0u;            // OR of the bits below this level
      sm->ubc[5] = 0xFFFFFFFFu;   // AND of the bits below this level
    }
    __syncthreads();
    uint32_t lo_or = 0u, lo_and = 0xFFFFFFFFu;
    visit([&](uint32_t key) {
      if (key != 0u && (key & mask) == prefix) {
        atomicAdd(&sm->hist[(key >> shift) & static_cast<uint32_t>(nb - 1)], 1u);
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
    find_bin(sm->hist, nb, need, sm, bin, above, cur);
    prefix |= static_cast<uint32_t>(bin) << shift;
    mask |= static_cast<uint32_t>(nb - 1) << shift;
    need -= above;
    if (all_or == (all_and & low)) {
      // every key still in play has the same lower bits: T is resolved
      prefix |= all_or;
      mask |= low;
      break;
    }
    hb = shift - 1;
  }
}

// Over the coarse sample histogram hist[b] (b = key >> 21): cbU = the smallest bin with
// cum(b) <= rU (2048: none; cum(b) = sample keys in bins >= b), cumU = cum(cbU); cbL = the
// largest bin with cum(b) >= rL (-1: none), cumL1 = cum(cbL + 1).
template <class SM>
__device__ __forceinline__ void coarse_window(int rU, int rL, int& cbU, int& cbL, int& cumU,
                                              int& cumL1, SM* sm) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    sm->bcast[0] = 2048;
    sm->bcast[1] = 0;
    sm->bcast[2] = -1;
    sm->bcast[3] = 0;
  }
  int c[8], sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = static_cast<int>(sm->hist[2047 - (8 * tid + j)]);
    sum += c[j];
  }
  int tot;
  int run = block_scan(sum, tot, sm) - sum;   // cum of the bins above this thread's
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int bb = 2047 - (8 * tid + j);
    const int cum = run + c[j];
    // cum(bb) <= rU < cum(bb - 1): bb is the smallest such bin
    if (cum <= rU) {
      const int next = bb > 0 ? static_cast<int>(sm->hist[bb - 1]) : 0;
      if (bb == 0 || cum + next > rU) {
        sm->bcast[0] = bb;
        sm->bcast[1] = cum;
      }
    }
    if (run < rL && cum >= rL) {
      sm->bcast[2] = bb;
      sm->bcast[3] = run;
    }
    run = cum;
  }
  __syncthreads();
  cbU = sm->bcast[0];
  cumU = sm->bcast[1];
  cbL = sm->bcast[2];
  cumL1 = sm->bcast[3];
  __syncthreads();
}

// From the fine histograms (hist[0,1024): bits 20..11 of the keys in coarse bin cbU - 1;
// hist[1024,2048): of those in coarse bin cbL): U = the lowest fine edge in bin cbU - 1
// with at most rU sample keys at or above it (else the coarse edge of cbU), L = the
// highest fine edge in bin cbL with at least rL (0 when there is no such bin).
template <class SM>
__device__ __forceinline__ void fine_window(int rU, int rL, int cbU, int cbL, int cumU, int cumL1,
                                            uint32_t& U, uint32_t& L, SM* sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool lhalf = tid >= NT / 2;   // threads of the L half
  const int h0 = lhalf ? 1024 : 0;
  const int t8 = (tid & (NT / 2 - 1)) * 8;   // 8 fine bins per thread, from the top
  if (tid == 0) {
    sm->bcast[0] = -1;
    sm->bcast[1] = -1;
  }
  int c[8], sum = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = static_cast<int>(sm->hist[h0 + 1023 - (t8 + j)]);
    sum += c[j];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm->warp_tot[warp] = incl;
  __syncthreads();
  int before = 0;
  for (int w = lhalf ? NW / 2 : 0; w < warp; ++w) before += sm->warp_tot[w];
  int run = before + incl - sum + (lhalf ? cumL1 : cumU);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int fb = 1023 - (t8 + j);
    const int cum = run + c[j];
    if (!lhalf) {
      // the smallest fine bin of coarse bin cbU - 1 with cum <= rU
      if (cbU >= 1 && cum <= rU) {
        const int next = fb > 0 ? static_cast<int>(sm->hist[fb - 1]) : rU + 1;
        if (cum + next > rU) sm->bcast[0] = fb;
      }
    } else if (cbL >= 0 && run < rL && cum >= rL) {
      sm->bcast[1] = fb;
    }
    run = cum;
  }
  __syncthreads();
  const int fu = sm->bcast[0], fl = sm->bcast[1];
  U = cbU >= 2048 ? 0xFFFFFFFFu : static_cast<uint32_t>(cbU) << 21;
  if (fu >= 0) U = (static_cast<uint32_t>(cbU - 1) << 21) | (static_cast<uint32_t>(fu) << 11);
  L = cbL < 0 ? 0u : static_cast<uint32_t>(cbL) << 21;
  if (fl >= 0) L |= static_cast<uint32_t>(fl) << 11;
  __syncthreads();
}

__global__ void __launch_bounds__(NT, 6) topk_short_kernel(const TopkParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  if (gated_off(p)) return;
  Smem* sm = reinterpret_cast<Smem*>(smem_raw);
  // rows t_lo <= t < min(t_hi, kStageMax) of every batch row, longest first
  const int nsc = min(p.t_hi, kStageMax) - p.t_lo;
  const long long i = static_cast<long long>(gridDim.x) - 1 - blockIdx.x;
  const int b = static_cast<int>(i / nsc);
  const int t = p.t_lo + static_cast<int>(i - static_cast<long long>(b) * nsc);
  const long long row = static_cast<long long>(b) * p.S + t;
  const int len = t + 1, nq = (len + 3) >> 2, nwords = (len + 31) >> 5;
  const int tid = threadIdx.x, lane = tid & 31;
  const int32_t* seg_row = p.seg ? p.seg + static_cast<long long>(b) * p.S : nullptr;
  const int seg_t = seg_row ? seg_row[t] : 0;
  const Row rk{score_row(p, b, t), seg_row, len, seg_t,
               (reinterpret_cast<uintptr_t>(seg_row) & 15u) == 0};
  int32_t* out = p.idx + row * p.k;
  float* vout = p.vals ? p.vals + row * p.k : nullptr;

  // number of valid keys
  int n = len;
  if (seg_row) {
    int c = 0;
    for (int q = tid; q < nq; q += NT) c += __popc(rk.valid4(q));
    int tot;
    block_scan(c, tot, sm);
    n = tot;
  }

  if (n <= p.k) {
    // every valid key is selected, in ascending order
    if (!seg_row) {
      for (int j = tid; j < p.k; j += NT) {
        out[j] = j < len ? j : -1;
        if (vout) vout[j] = j < len ? __ldg(rk.srow + j) : -INFINITY;
      }
    } else {
      for (int c0 = 0; c0 < nq; c0 += NT) {
        const int c = c0 + tid;
        const uint32_t wv = gather_word(c < nq ? rk.valid4(c) : 0u, lane);
        if ((lane & 7) == 0 && c < nq) {
          sm->gtw[c >> 3] = wv;
          sm->eqw[c >> 3] = 0u;
        }
      }
      __syncthreads();
      if (vout)
        emit<true>(nwords, 0, n, out, p.k, sm, rk.srow, vout);
      else
        emit<false>(nwords, 0, n, out, p.k, sm, rk.srow, vout);
    }
    if (p.count && tid == 0) p.count[row] = n;
    return;
  }

  // ---- sample: eight keys per thread (two groups of four), spread over the row, or
  // every group once when the row has at most 2 * NT of them
  uint32_t sk[kSampleGroups][4];
  const bool full = nq <= kSampleGroups * NT;
#pragma unroll
  for (int j = 0; j < kSampleGroups; ++j) {
    const int c = full ? tid + NT * j
                       : static_cast<int>((static_cast<long long>(tid + NT * j) * nq) /
                                          (kSampleGroups * NT));
    if (c < nq) {
      rk.load4(c, sk[j]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) sk[j][e] = 0u;
    }
  }
  for (int j = tid; j < 2048; j += NT) sm->hist[j] = 0u;
  if (tid == 0) {
    for (int j = 0; j < 8; ++j) sm->ubc[j] = 0u;
  }
  __syncthreads();
  // coarse level: 2048 bins of key >> 21 (sign, exponent, two mantissa bits) over the
  // whole key range, so the window may hold T on either side of zero
  int nvalid = 0;
#pragma unroll
  for (int j = 0; j < kSampleGroups; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (sk[j][e] != 0u) {
        atomicAdd(&sm->hist[sk[j][e] >> 21], 1u);
        ++nvalid;
      }
  nvalid = __reduce_add_sync(0xffffffffu, nvalid);
  if (lane == 0) atomicAdd(&sm->ubc[3], static_cast<uint32_t>(nvalid));
  __syncthreads();
  const uint32_t ns = sm->ubc[3];
  // sample ranks bracketing T: rank r = k * ns / n from the top, +- kZ sigma (binomial,
  // with the finite-population factor: a full sample gives the exact rank)
  const float pk = static_cast<float>(p.k) / static_cast<float>(n);
  const float fr = static_cast<float>(ns) / static_cast<float>(n);
  const float r = pk * static_cast<float>(ns);
  const float sd = sqrtf(fmaxf(static_cast<float>(ns) * pk * (1.f - pk) * (1.f - fr), 0.f));
  const int rU = static_cast<int>(floorf(r - kZ * sd));   // keys >= U: likely all selected
  const int rL = static_cast<int>(ceilf(r + kZ * sd));    // keys >= L: likely at least k
  int cbU, cbL, cumU, cumL1;
  coarse_window(rU, rL, cbU, cbL, cumU, cumL1, sm);
  // fine level: 1024 bins of bits 20..11 inside the coarse bin just below U (hist[0,1024))
  // and inside the coarse bin of L (hist[1024,2048)), to place U and L 2^11 keys apart
  for (int j = tid; j < 2048; j += NT) sm->hist[j] = 0u;
  __syncthreads();
  const int cu = cbU - 1;   // the coarse bin below U (-1: none)
#pragma unroll
  for (int j = 0; j < kSampleGroups; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t kk = sk[j][e];
      if (kk == 0u) continue;
      const int cb = static_cast<int>(kk >> 21);
      const uint32_t fb = (kk >> 11) & 1023u;
      if (cb == cu) atomicAdd(&sm->hist[fb], 1u);
      if (cb == cbL) atomicAdd(&sm->hist[1024 + fb], 1u);
    }
  __syncthreads();
  uint32_t U, L;
  fine_window(rU, rL, cbU, cbL, cumU, cumL1, U, L, sm);
  for (int w = tid; w < nwords; w += NT) sm->eqw[w] = 0u;

  // ---- one sweep: keys >= U into gtw (counted), keys in [L, U) into the list. The tests
  // run on the raw scores against L and U as floats (the order map is monotone, and an
  // invalid key is read as NaN, which fails every comparison); only listed keys are
  // mapped to order keys.
  const float fU = key_to_float(U), fL = key_to_float(L);
  int cnt_above = 0;
  // kSweepDepth groups of four per thread in flight per step (one DRAM latency per step)
  for (int c0 = 0; c0 < nq; c0 += kSweepDepth * NT) {
    float f[kSweepDepth][4];
#pragma unroll
    for (int u = 0; u < kSweepDepth; ++u) {
      const int c = c0 + u * NT + tid;
#pragma unroll
      for (int e = 0; e < 4; ++e) f[u][e] = __int_as_float(0x7fc00000);
      if (c < nq) rk.load4f(c, f[u]);
    }
#pragma unroll
    for (int u = 0; u < kSweepDepth; ++u) {
      const int c = c0 + u * NT + tid;
      uint32_t nib = 0u, cm = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        nib |= static_cast<uint32_t>(f[u][e] >= fU) << e;
        cm |= static_cast<uint32_t>(f[u][e] >= fL && !(f[u][e] >= fU)) << e;
      }
      cnt_above += __popc(nib);
      const uint32_t wv = gather_word(nib, lane), wc = gather_word(cm, lane);
      if ((lane & 7) == 0 && c < nq) {
        sm->gtw[c >> 3] = wv;
        sm->cw[c >> 3] = wc;
      }
    }
  }
  cnt_above = __reduce_add_sync(0xffffffffu, cnt_above);
  if (lane == 0) atomicAdd(&sm->ubc[7], static_cast<uint32_t>(cnt_above));
  __syncthreads();   // gtw, cw and the count are complete
  // the window keys, from their bitmap, into the list in ascending index: the indices
  // first, then their order keys from scores the sweep left in L2, read by every thread
  // in turn so that the loads overlap instead of following each thread's bits
  uint32_t cwv[kWpt];
  int cc = 0;
#pragma unroll
  for (int i = 0; i < kWpt; ++i) {
    const int w = kWpt * tid + i;
    cwv[i] = w < nwords ? sm->cw[w] : 0u;
    cc += __popc(cwv[i]);
  }
  int ncand;
  int slot = block_scan(cc, ncand, sm) - cc;
  const int A = static_cast<int>(sm->ubc[7]);
  if (ncand <= kCand) {
#pragma unroll
    for (int i = 0; i < kWpt; ++i) {
      uint32_t m = cwv[i];
      while (m) {
        const int bpos = __ffs(m) - 1;
        m &= m - 1u;
        sm->cidx[slot++] = static_cast<uint16_t>((kWpt * tid + i) * 32 + bpos);
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int j = tid; j < ncand; j += NT) sm->ckey[j] = order_key(__ldg(rk.srow + sm->cidx[j]));
  }
  __syncthreads();

  uint32_t prefix = 0u, mask = 0u;
  int need = p.k;
  if (A <= p.k && A + ncand >= p.k && ncand <= kCand) {
    // T is in the list: its digits below the common prefix of L and U - 1
    need = p.k - A;
    if (need > 0) {
      const uint32_t d = L ^ (U - 1u);
      const int hb = d == 0u ? -1 : 31 - __clz(d);
      mask = hb < 0 ? 0xFFFFFFFFu : (hb >= 31 ? 0u : ~((2u << hb) - 1u));
      prefix = L & mask;
      resolve([&](auto fn) {
        for (int j = tid; j < ncand; j += NT) fn(sm->ckey[j]);
      }, hb, prefix, mask, need, ncand, sm, 8);
      // list keys above T / equal to T into the bitmaps
      for (int j = tid; j < ncand; j += NT) {
        const uint32_t km = sm->ckey[j] & mask;
        const int s = sm->cidx[j];
        if (km > prefix) atomicOr(&sm->gtw[s >> 5], 1u << (s & 31));
        else if (km == prefix) atomicOr(&sm->eqw[s >> 5], 1u << (s & 31));
      }
      __syncthreads();
    }
  } else {
    // the window missed (or its list overflowed): radix select over the whole row,
    // then both bitmaps from one more sweep
    resolve([&](auto fn) {
      for (int c = tid; c < nq; c += NT) {
        uint32_t kq[4];
        rk.load4(c, kq);
#pragma unroll
        for (int e = 0; e < 4; ++e) fn(kq[e]);
      }
    }, 31, prefix, mask, need, n, sm);
    for (int c0 = 0; c0 < nq; c0 += NT) {
      const int c = c0 + tid;
      uint32_t kq[4] = {0u, 0u, 0u, 0u};
      if (c < nq) rk.load4(c, kq);
      uint32_t ng = 0u, ne = 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t km = kq[e] & mask;
        ng |= static_cast<uint32_t>(kq[e] != 0u && km > prefix) << e;
        ne |= static_cast<uint32_t>(kq[e] != 0u && km == prefix) << e;
      }
      const uint32_t wg = gather_word(ng, lane), we = gather_word(ne, lane);
      if ((lane & 7) == 0 && c < nq) {
        sm->gtw[c >> 3] = wg;
        sm->eqw[c >> 3] = we;
      }
    }
    __syncthreads();
  }
  if (vout)
    emit<true>(nwords, need, p.k, out, p.k, sm, rk.srow, vout);
  else
    emit<false>(nwords, need, p.k, out, p.k, sm, rk.srow, vout);
  if (p.count && tid == 0) p.count[row] = p.k;
}

}  // namespace sr

// ------------------------------------------------------- streaming form (no score rows)
// The indexer's sample pass leaves, per query row, the scores of sample_tiles(nkb) evenly
// spaced 128-key tiles of its query group's causal range (NaN where a key is not valid).
// stream_window_kernel turns them into the row's window [L, U) as floats, exactly as the
// short-row kernel does with its own sample. The indexer's emit pass then lists every
// valid key scoring >= U (into the row's idx slots, unordered) and every key in [L, U)
// (index and score) without storing any other score. stream_finish_kernel settles the row
// from the two lists, or flags its block of rows for the memory form.
namespace st {

constexpr int NT = 256;
constexpr int NW = NT / 32;
constexpr int kMaxS = kStreamMaxS;       // keys per row (bitmaps of kMaxS bits)
constexpr int kWords = kMaxS / 32;
constexpr int kCw = kStreamWindowCap;    // window keys per row
// window half-width in standard deviations: a row the window misses costs its whole
// block of rows, so the odds of a miss are kept near 1e-6 per row
constexpr float kZ = 5.f;

struct WinSmem {
  uint32_t hist[2048];
  int warp_tot[NW];
  int bcast[4];
  uint32_t ubc[8];
};

struct FinSmem {
  uint32_t hist[2048];       // level histograms, then the output row
  uint32_t gtw[kWords];      // keys above T (with vals: then the selected keys of each word)
  uint32_t eqw[kWords];      // keys equal to T
  uint32_t ckey[kCw];        // window keys: order key
  int32_t cidx[kCw];         //   and index
  int wbase[kWords];         // with vals: the first slot of each word's selected keys
  float vst[2048];           // with vals: the row's selected scores by slot
  int warp_tot[NW];
  int bcast[4];
  uint32_t ubc[8];
};

// one CTA per row: (U, L) as floats from the row's sample, NaN for rows that need none
__global__ void __launch_bounds__(NT) stream_window_kernel(const float* sample, int B, int S,
                                                           int G, int k, float* thr) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  WinSmem* sm = reinterpret_cast<WinSmem*>(smem_raw);
  const long long row = blockIdx.x;
  const int t = static_cast<int>(row % S);
  const int tid = threadIdx.x, lane = tid & 31;
  if (t + 1 <= k) {   // at most k valid keys: all of them are selected (U = L = -inf)
    if (tid == 0) {
      thr[2 * row] = -INFINITY;
      thr[2 * row + 1] = -INFINITY;
    }
    return;
  }
  // the sampled tiles of the row's query group (as the indexer's sample pass chose them)
  const int t0 = (t / G) * G, t_last = min(t0 + G - 1, S - 1);
  const int nkb = t_last / 128 + 1, nt = sample_tiles(nkb);
  const float* srow = sample + row * kSampleKeys;
  uint32_t sk[kSampleKeys / NT];
  int causal = 0;   // sampled slots with key <= t
#pragma unroll
  for (int j = 0; j < kSampleKeys / NT; ++j) {
    const int slot = tid + NT * j, m = slot >> 7;
    sk[j] = 0u;
    if (m < nt) {
      const int key = sample_tile(m, nt, nkb) * 128 + (slot & 127);
      causal += key <= t;
      const float v = srow[slot];
      if (v == v) sk[j] = order_key(v);   // NaN: not a valid key
    }
  }
  for (int j = tid; j < 2048; j += NT) sm->hist[j] = 0u;
  if (tid == 0)
    for (int j = 0; j < 8; ++j) sm->ubc[j] = 0u;
  __syncthreads();
  int nvalid = 0;
#pragma unroll
  for (int j = 0; j < kSampleKeys / NT; ++j)
    if (sk[j] != 0u) {
      atomicAdd(&sm->hist[sk[j] >> 21], 1u);
      ++nvalid;
    }
  nvalid = __reduce_add_sync(0xffffffffu, nvalid);
  causal = __reduce_add_sync(0xffffffffu, causal);
  if (lane == 0) {
    atomicAdd(&sm->ubc[3], static_cast<uint32_t>(nvalid));
    atomicAdd(&sm->ubc[4], static_cast<uint32_t>(causal));
  }
  __syncthreads();
  const uint32_t ns = sm->ubc[3], nc = sm->ubc[4];
  // valid keys of the row: t + 1 without documents; with documents estimated from the
  // sample's share of valid keys among its causal ones (only the window depends on it)
  const float n = nc > 0 ? static_cast<float>(t + 1) * static_cast<float>(ns) / static_cast<float>(nc)
                         : static_cast<float>(t + 1);
  const float pk = fminf(static_cast<float>(k) / fmaxf(n, 1.f), 1.f);
  const float fr = fminf(static_cast<float>(ns) / fmaxf(n, 1.f), 1.f);
  const float r = pk * static_cast<float>(ns);
  const float sd = sqrtf(fmaxf(static_cast<float>(ns) * pk * (1.f - pk) * (1.f - fr), 0.f));
  const int rU = static_cast<int>(floorf(r - kZ * sd));
  const int rL = static_cast<int>(ceilf(r + kZ * sd));
  int cbU, cbL, cumU, cumL1;
  sr::coarse_window(rU, rL, cbU, cbL, cumU, cumL1, sm);
  for (int j = tid; j < 2048; j += NT) sm->hist[j] = 0u;
  __syncthreads();
  const int cu = cbU - 1;
#pragma unroll
  for (int j = 0; j < kSampleKeys / NT; ++j) {
    const uint32_t kk = sk[j];
    if (kk == 0u) continue;
    const int cb = static_cast<int>(kk >> 21);
    const uint32_t fb = (kk >> 11) & 1023u;
    if (cb == cu) atomicAdd(&sm->hist[fb], 1u);
    if (cb == cbL) atomicAdd(&sm->hist[1024 + fb], 1u);
  }
  __syncthreads();
  uint32_t U, L;
  sr::fine_window(rU, rL, cbU, cbL, cumU, cumL1, U, L, sm);
  if (tid == 0) {
    thr[2 * row] = sr::key_to_float(U);
    thr[2 * row + 1] = sr::key_to_float(L);
  }
}

// the keys > T (gtw) and the lowest-index `need` keys == T (eqw), `total` in all, into
// out[0, total) ascending and -1 into out[total, kmax); each thread owns a contiguous run
// of `per` bitmap words. With vals (kmax <= 2048) each slot's score as well: the keys
// >= U have theirs beside the unordered list in out[0, A) / vals[0, A) (the emit pass
// wrote them there), the window keys in wrow[0, W); each goes to its key's slot.
__device__ __forceinline__ void emit_words(int nwords, int need, int total, int32_t* out,
                                           int kmax, FinSmem* sm, float* vals, int A,
                                           const int2* wrow, int W) {
  const int tid = threadIdx.x;
  const int per = (nwords + NT - 1) / NT;
  const int w0 = min(tid * per, nwords), w1 = min(w0 + per, nwords);
  int cg = 0, ce = 0;
  for (int w = w0; w < w1; ++w) {
    cg += __popc(sm->gtw[w]);
    ce += __popc(sm->eqw[w]);
  }
  const int own = cg | (ce << 16);
  int tot;
  const int excl = sr::block_scan(own, tot, sm) - own;
  int eb = excl >> 16;
  int pos = (excl & 0xFFFF) + min(eb, need);
  int32_t* ost = kmax <= 2048 ? reinterpret_cast<int32_t*>(sm->hist) : out;
  for (int w = w0; w < w1; ++w) {
    const uint32_t q = sm->eqw[w];
    uint32_t qk = 0u, m = q;
    for (int room = need - eb; m != 0u && room > 0; --room) {
      const uint32_t low = m & (0u - m);
      qk |= low;
      m ^= low;
    }
    eb += __popc(q);
    uint32_t sel = sm->gtw[w] | qk;
    if (vals) {   // only this thread reads its words from here on
      sm->wbase[w] = pos;
      sm->gtw[w] = sel;
    }
    while (sel) {
      const int bpos = __ffs(sel) - 1;
      sel &= sel - 1u;
      if (pos < kmax) ost[pos] = w * 32 + bpos;
      ++pos;
    }
  }
  if (ost != out) {
    __syncthreads();
    if (vals) {
      // a selected key's slot: its word's first slot plus the selected keys below it
      auto slot = [&](int key) {
        const uint32_t m = sm->gtw[key >> 5], bit = 1u << (key & 31);
        return (m & bit) ? sm->wbase[key >> 5] + __popc(m & (bit - 1u)) : -1;
      };
      for (int j = tid; j < A; j += NT) {
        const int q = slot(out[j]);
        if (q >= 0 && q < kmax) sm->vst[q] = vals[j];
      }
      for (int j = tid; j < W; j += NT) {
        const int2 e = wrow[j];
        const int q = slot(e.x);
        if (q >= 0 && q < kmax) sm->vst[q] = __int_as_float(e.y);
      }
      __syncthreads();   // every old entry of out / vals is read before they are rewritten
    }
    for (int j = tid; j < kmax; j += NT) {
      out[j] = j < total ? ost[j] : -1;
      if (vals) vals[j] = j < total ? sm->vst[j] : -INFINITY;
    }
  } else {   // (kmax > 2048: never with vals)
    for (int j = total + tid; j < kmax; j += NT) out[j] = -1;
  }
}

// one CTA per row, longest rows first
__global__ void __launch_bounds__(NT) stream_finish_kernel(const int32_t* seg, int B, int S, int k,
                                                           const int* cnt, const int2* win, int cw,
                                                           int32_t* idx, int32_t* count, float* vals,
                                                           int* flags, int block_rows) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  FinSmem* sm = reinterpret_cast<FinSmem*>(smem_raw);
  const long long i = static_cast<long long>(gridDim.x) - 1 - blockIdx.x;
  const int b = static_cast<int>(i / S), t = static_cast<int>(i % S);
  const long long row = i;
  const int len = t + 1, nwords = (len + 31) >> 5;
  const int tid = threadIdx.x;
  const int32_t* seg_row = seg ? seg + static_cast<long long>(b) * S : nullptr;
  const int seg_t = seg_row ? seg_row[t] : 0;
  int32_t* out = idx + row * k;
  float* vout = vals ? vals + row * k : nullptr;
  (void)seg_t;
  for (int w = tid; w < nwords; w += NT) {
    sm->gtw[w] = 0u;
    sm->eqw[w] = 0u;
  }
  __syncthreads();
  // (rows of at most k keys have U = -inf: their every valid key is in the list >= U)
  const int A = cnt[4 * row], W = cnt[4 * row + 1];
  const int n = seg_row ? cnt[4 * row + 2] : len;
  const int m = n < k ? n : k;   // keys to select
  const bool settled = A <= m && W <= cw && (n <= k ? A + W == n : A + W >= k);
  if (!settled) {
    // the sampled window missed this row: the memory form redoes its block of rows
    if (tid == 0) flags[t / block_rows] = 1;
    return;
  }
  // the keys >= U (written unordered into the row's own idx slots by the emit pass)
  const int above_n = A;
  for (int j = tid; j < above_n; j += NT) {
    const int s = out[j];
    atomicOr(&sm->gtw[s >> 5], 1u << (s & 31));
  }
  for (int j = tid; j < W; j += NT) {
    const int2 e = win[row * cw + j];
    sm->cidx[j] = e.x;
    sm->ckey[j] = order_key(__int_as_float(e.y));
  }
  if (tid == 0)
    for (int j = 0; j < 8; ++j) sm->ubc[j] = 0u;
  __syncthreads();
  int need = m - A;
  if (need > 0 && W == need) {
    for (int j = tid; j < W; j += NT) atomicOr(&sm->gtw[sm->cidx[j] >> 5], 1u << (sm->cidx[j] & 31));
    need = 0;
    __syncthreads();
  } else if (need > 0) {
    // T among the window keys: every listed key lies in [L, U), so radix over all 32 bits
    uint32_t prefix = 0u, mask = 0u;
    sr::resolve([&](auto fn) {
      for (int j = tid; j < W; j += NT) fn(sm->ckey[j]);
    }, 31, prefix, mask, need, W, sm, 8);
    for (int j = tid; j < W; j += NT) {
      const uint32_t km = sm->ckey[j] & mask;
      const int s = sm->cidx[j];
      if (km > prefix) atomicOr(&sm->gtw[s >> 5], 1u << (s & 31));
      else if (km == prefix) atomicOr(&sm->eqw[s >> 5], 1u << (s & 31));
    }
    __syncthreads();
  }
  emit_words(nwords, need, m, out, k, sm, vout, A, win + row * cw, W);
  if (count && tid == 0) count[row] = m;
}

}  // namespace st

// ------------------------------------------------------------------ long rows
// Rows longer than the shared stage (t >= kStageMax): two persistent CTAs of 512
// threads per SM, each on its own row, so that one row's barrier-bound phases (the
// sample, the bins, the list and the emission) overlap the other's pass over its
// keys; each row is prefetched whole into L2 (304 rows in flight, at most 512 KB
// each at S = 131072). Every pass reads the row from global memory in 16-byte
// groups of four keys. The selection is the same as for staged rows: a window
// histogram, then either a candidate list with bitmaps (rows of at most
// kLongWords * 32 keys and at most kLongCand keys in the threshold bin) or further
// levels over the row with an ordered sweep.
namespace lr {

constexpr int NT = 512;
constexpr int NW = NT / 32;
constexpr int kLongWords = 4096;   // bitmap words: rows up to 131072 keys
// candidates of the one-pass path: each warp appends to its own segment of 512; at
// S = 131072 the 2048-key sample leaves a row about 4K candidates, ~250 per warp
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

// the bin of the need-th largest key among nb bins (nb <= 2048), keys above it
// and in it
__device__ __forceinline__ void find_bin(const uint32_t* hist, int nb, int need, Smem* sm,
                                         int& bin, int& above, int& in_bin) {
  const int per = nb > NT ? nb / NT : 1;
  const int tid = threadIdx.x;
  constexpr int kPer = (2048 + NT - 1) / NT;
  int c[kPer];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int j = tid * per + i;
    c[i] = i < per && j < nb ? static_cast<int>(hist[nb - 1 - j]) : 0;
    sum += c[i];
  }
  int tot;
  const int incl = block_scan(sum, tot, sm);
  int run = incl - sum;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
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
// Up to four digit levels (shift, number of bins) held in registers: selected by constant
// index, so that no table lands in local memory, where streaming rows would evict it to DRAM.
struct Levels {
  int n, s0, s1, s2, s3, b0, b1, b2, b3;
  __device__ __forceinline__ int shift(int l) const {
    return l == 0 ? s0 : (l == 1 ? s1 : (l == 2 ? s2 : s3));
  }
  __device__ __forceinline__ int bins(int l) const {
    return l == 0 ? b0 : (l == 1 ? b1 : (l == 2 ? b2 : b3));
  }
};

template <class Visit>
__device__ __forceinline__ void resolve_levels(Visit visit, uint32_t* hist, const Levels lv,
                                               uint32_t& prefix, uint32_t& mask, int& need,
                                               int in_bin, Smem* sm) {
  const int tid = threadIdx.x, lane = tid & 31;
#pragma unroll 1
  for (int lvl = 0; lvl < lv.n && in_bin != need; ++lvl) {
    const int shift = lv.shift(lvl), nb = lv.bins(lvl);
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
  const Levels lv_in = {2, 8, 0, 0, 0, 512, 256, 0, 0};
  const Levels lv_out = {4, 24, 16, 8, 0, 256, 256, 256, 256};
  resolve_levels(
      [&](auto fn) {
        for (int j = tid; j < ncand; j += NT) fn(rk.key(static_cast<int>(sm->cand[j])));
      },
      sm->hist, inner ? lv_in : lv_out, prefix, mask, need, in_bin, sm);
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
  // the first group of each thread (the row's first 4 * NT keys) places the window
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
    const Levels lv_in = {2, 6, 0, 0, 0, 2048, 64, 0, 0};
    const Levels lv_out = {3, 21, 10, 0, 0, 2048, 2048, 1024, 0};
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
        sm->hist, inner ? lv_in : lv_out, prefix, mask, need, in_bin, sm);
    select_sweep(rk, nq, mask, prefix, need, out, p.k, sm);
  }
  if (p.count && tid == 0) p.count[row] = p.k;
  __syncthreads();   // the shared state is reused by the next row
}

}  // namespace lr

// rows t0 <= t < t_hi of every batch row; persistent, longest rows first, two CTAs per SM
__global__ void __launch_bounds__(lr::NT, 2) topk_long_kernel(const TopkParams p, int t0) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  if (gated_off(p)) return;
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
    {
      // the whole row into L2 ahead of its passes (16 KB per bulk prefetch, one per
      // thread): the sample's round trip and the later passes then overlap its transfer
      const long long bytes = static_cast<long long>((t + 4) >> 2) * 16;
      const long long c0 = static_cast<long long>(tid) * 16384;
      if (c0 < bytes) {
        const long long sz = bytes - c0 < 16384 ? bytes - c0 : 16384;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                         reinterpret_cast<const char*>(rk.srow) + c0),
                     "r"(static_cast<uint32_t>(sz))
                     : "memory");
      }
    }
    lr::select_row(rk, t, n, p, p.idx + row * p.k, row, sm);
    if (p.vals) {
      // the row's slots are written (by every thread, in whichever path selected them):
      // their scores, while the row is in L2
      __syncthreads();
      const int32_t* o = p.idx + row * p.k;
      float* v = p.vals + row * p.k;
      for (int j = tid; j < p.k; j += lr::NT) {
        const int s = __ldcg(o + j);
        v[j] = s >= 0 ? __ldg(rk.srow + s) : -INFINITY;
      }
    }
  }
}
}  // namespace

int launch_topk(const float* scores, int64_t ld, const int32_t* seg, int B, int S, int k,
                int32_t* idx, int32_t* count, float* vals, cudaStream_t stream) {
  return launch_topk_rows(scores, ld, seg, B, S, k, idx, count, vals, stream, 0, S, S);
}

int launch_topk_rows(const float* scores, int64_t ld, const int32_t* seg, int B, int S, int k,
                     int32_t* idx, int32_t* count, float* vals, cudaStream_t stream, int t_lo,
                     int t_hi, long long rows_blk, const int* gate) {
  TopkParams p;
  p.gate = gate;
  p.vals = vals;
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
  const long long rows = static_cast<long long>(B) * S;
  if (rows > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
  // rows t < kStageMax: one CTA of sr::NT threads per row
  const int short_hi = t_hi < kStageMax ? t_hi : kStageMax;
  if (short_hi > t_lo) {
    const size_t smem = sizeof(sr::Smem);
    if (cudaFuncSetAttribute(sr::topk_short_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return DSA_ERR_CUDA;
    const long long nshort = static_cast<long long>(B) * (short_hi - t_lo);
    sr::topk_short_kernel<<<static_cast<unsigned>(nshort), sr::NT, smem, stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  }
  const int long_lo = t_lo > kStageMax ? t_lo : kStageMax;
  if (S > kStageMax && t_hi > long_lo) {
    // longer rows: persistent CTAs, two per SM
    const size_t lsmem = sizeof(lr::Smem);
    if (cudaFuncSetAttribute(topk_long_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(lsmem)) != cudaSuccess)
      return DSA_ERR_CUDA;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long nlong = static_cast<long long>(B) * (t_hi - long_lo);
    const int grid = static_cast<int>(nlong < 2 * sms ? nlong : 2 * sms);
    topk_long_kernel<<<grid, lr::NT, lsmem, stream>>>(p, long_lo);
    if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;
  }
  return DSA_OK;
}

int launch_stream_window(const float* sample, const int32_t* seg, int B, int S, int G, int k,
                         float* thr, cudaStream_t stream) {
  (void)seg;
  const long long rows = static_cast<long long>(B) * S;
  if (rows > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
  st::stream_window_kernel<<<static_cast<unsigned>(rows), st::NT, sizeof(st::WinSmem), stream>>>(
      sample, B, S, G, k, thr);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

int launch_stream_finish(const int32_t* seg, int B, int S, int k, const int* cnt,
                         const int2* win, int cw, int32_t* idx, int32_t* count, float* vals,
                         int* flags, int block_rows, cudaStream_t stream) {
  if (S > st::kMaxS || cw > st::kCw) return DSA_ERR_UNSUPPORTED;
  if (vals && k > 2048) return DSA_ERR_UNSUPPORTED;   // the scores are staged by slot
  const long long rows = static_cast<long long>(B) * S;
  if (rows > 0x7fffffffLL) return DSA_ERR_UNSUPPORTED;
  const size_t smem = sizeof(st::FinSmem);
  if (cudaFuncSetAttribute(st::stream_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  st::stream_finish_kernel<<<static_cast<unsigned>(rows), st::NT, smem, stream>>>(
      seg, B, S, k, cnt, win, cw, idx, count, vals, flags, block_rows);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
