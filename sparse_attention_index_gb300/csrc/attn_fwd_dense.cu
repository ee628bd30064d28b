// Sparse attention forward on dense 128 x 128 tiles with a selection bitmap.
//
// ("Support Ring Attention with DeepSeek DSA Sparse Indexer", Forward Flow step 5:
// logits = where(mask, Q K^T * scale, -inf); the pages evaluate this as dense
// blocks with partial mask blocks. Here that is the path for few heads and many
// selected keys per query, where the gathered-key kernel, which puts the heads on
// the M = 128 lanes, would leave most of each tile idle.)
//
// One work item is (batch b, head h, tile of 128 query rows). Each TMEM lane is one
// query row, so the M = 128 tile is full whatever H is:
//   S  = Q_tile [128 x Dqk] . K_tile^T       A = Q from TMEM, B = K tile in smem (K-major)
//   P  = exp2(S * scale*log2e - m) where the row selects the key, else 0
//   O += P [128 x 128] . V_tile [128 x Dv]   A = P from TMEM, B = V tile in smem (MN-major)
// The selection is a bitmap built from the index lists (dense_mask_kernel): bit s of
// row t is set when row t lists key s (0 <= s <= t); a row's words past its own query
// tile are never written nor read. A key tile in which no row of
// the query tile selects anything is skipped; the others stream through a 2-stage
// TMA ring. The running max is refreshed only when it grows by more than 2^8 (in
// exp2 units), as in the gathered-key kernel.
//
// Persistent CTA (one per SM), 320 threads:
//   warp  0     TMA producer: the active key tiles of each item, K and V (128B swizzle)
//   warp  1     TMEM owner and single-thread UMMA issuer
//   warps 2-9   softmax / output: Q rows -> TMEM, masked softmax, P -> TMEM, final O, LSE;
//               two warps per TMEM lane quarter, each on half of a tile's keys and of
//               the O columns
// TMEM: [Q: Dqk/2 cols][S/P: 2 x 128 cols][O: Dv cols].
// Items are handed out heaviest (last query tile) first, strided over CTAs.

#include "dsa_attn_common.cuh"

namespace dsa {
namespace {

constexpr int kTile = 128;            // query rows and keys per tile
constexpr int kStages = 2;            // K/V stages == S/P buffers
constexpr int kSoftWarps = 8;
constexpr int kThreads = 32 * (2 + kSoftWarps);
constexpr int kSoftWarp0 = 2;
constexpr int kErrD = DSA_STAGE_FWD | DSA_DEVERR_TIMEOUT;
constexpr float kRescaleLog2D = 8.f;  // refresh the running max when it grows by > 2^8

template <int DQK, int DV>
struct DenseLayout {
  static constexpr int KA = DQK / 64;                 // K atoms (64 dims each)
  static constexpr int VA = DV / 64;                  // V atoms
  static constexpr uint32_t kAtom = kTile * 128;      // one [128 rows x 128 B] atom
  static constexpr uint32_t kStage = (KA + VA) * kAtom;
  static constexpr uint32_t kTailOff = kStages * kStage;
  static constexpr uint32_t kColQ = 0;
  static constexpr uint32_t kColS = DQK / 2;
  static constexpr uint32_t kColO = kColS + kStages * kTile;
  static_assert(kColO + DV <= 512, "TMEM budget");
};

struct DenseHdr {
  int b, h, qt, kt;
  int first, last;   // first / last key tile of the item
  int pad[2];
};

struct DenseTail {
  DenseHdr hdr[kStages];
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[kStages], s_empty[kStages], p_full[kStages];
  uint64_t q_full, o_free;
  uint64_t drain;
  float xmax[2][2][kTile];   // per tile parity and half: the half's row max
  float xl[2][kTile];        // per half: the row sum at the end of an item
  uint64_t pairbar[4];       // per TMEM lane quarter: the two warps' exchange barrier
  uint32_t tmem_base;
  int abort_flag;
};

struct DenseParams {
  AttnParams a;
  const uint32_t* bits;   // [B*S, W4] selection bitmap, W4 words per row
  const uint8_t* any;     // [B, QT, QT]: does any row of query tile qt select in key tile kt
  int W4, QT;
};

// Selection bitmap and tile flags from the index lists, one row per CTA at a time:
// the row's words are built in shared memory and written out whole up to the row's
// own query tile (the only words the attention kernel reads); the tile flags must be
// zero beforehand. Entries -1 and entries above the diagonal are skipped;
// out-of-range entries set the device error word and are skipped, as in the other
// attention kernels.
__global__ void __launch_bounds__(256) dense_mask_kernel(const int32_t* idx, int B, int S, int k,
                                                         int W4, int QT, uint32_t* bits,
                                                         uint8_t* any, int* err) {
  extern __shared__ __align__(16) uint32_t words[];   // W4 words
  const long long rows = static_cast<long long>(B) * S;
  for (long long row = blockIdx.x; row < rows; row += gridDim.x) {
    const int b = static_cast<int>(row / S);
    const int t = static_cast<int>(row - static_cast<long long>(b) * S);
    const int nw = ((t >> 7) + 1) * 4;   // words of the key tiles up to the row's own
    for (int w = threadIdx.x; w < nw; w += blockDim.x) words[w] = 0u;
    __syncthreads();
    const int32_t* ir = idx + row * k;
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
      const int s = __ldg(ir + j);
      if (s < -1 || s >= S) {
        report_error(err, DSA_STAGE_FWD | DSA_DEVERR_BAD_INDEX);
        continue;
      }
      if (s < 0 || s > t) continue;
      atomicOr(&words[s >> 5], 1u << (s & 31));
    }
    __syncthreads();
    uint4* dst = reinterpret_cast<uint4*>(bits + row * W4);
    uint8_t* arow = any + (static_cast<long long>(b) * QT + (t >> 7)) * QT;
    for (int q = threadIdx.x; q < nw / 4; q += blockDim.x) {
      const uint4 v = reinterpret_cast<const uint4*>(words)[q];
      dst[q] = v;
      if ((v.x | v.y | v.z | v.w) != 0u) arow[q] = 1;   // key tile q has a selected key
    }
    __syncthreads();
  }
}

__device__ __forceinline__ void item_of(int i, int B, int H, int QT, int& b, int& h, int& qt) {
  const int bh = B * H;
  qt = QT - 1 - i / bh;
  const int r = i - (QT - 1 - qt) * bh;
  b = r / H;
  h = r - b * H;
}

__device__ __forceinline__ void drain_wait_d(uint64_t* bar, uint32_t parity, int* err) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report_error(err, kErrD);
      return;
    }
  }
}

__device__ __forceinline__ float ex2d(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_ld_x16d(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_dense_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const DenseParams dp) {
  using L = DenseLayout<DQK, DV>;
  const AttnParams& p = dp.a;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) report_error(p.err, DSA_STAGE_FWD | DSA_DEVERR_MISALIGNED);
    return;
  }
  DenseTail* tail = reinterpret_cast<DenseTail*>(smem + L::kTailOff);
  volatile int* abort_flag = &tail->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.B, S = p.S, H = p.H, QT = dp.QT;
  const int nitems = QT * B * H;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&tail->kv_full[i], 1);
      mbar_init(&tail->kv_empty[i], 1);
      mbar_init(&tail->s_full[i], 1);
      mbar_init(&tail->s_empty[i], 1);
      mbar_init(&tail->p_full[i], 32 * kSoftWarps);
    }
    mbar_init(&tail->q_full, 32 * kSoftWarps);
    mbar_init(&tail->o_free, 32 * kSoftWarps);
    mbar_init(&tail->drain, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&tail->pairbar[q], 64);
    tail->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&tail->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tail->tmem_base;

  if (warp == 0) {
    // ================================================================ TMA producer
    // The lanes scan the item's tile flags 32 at a time; lane 0 issues the copies.
    int g = 0;
    bool ok = true;
    uint32_t last_par[kStages] = {0, 0};
    bool issued[kStages] = {false, false};
    for (int i = blockIdx.x; ok && i < nitems; i += gridDim.x) {
      int b, h, qt;
      item_of(i, B, H, QT, b, h, qt);
      const uint8_t* arow = dp.any + (static_cast<long long>(b) * QT + qt) * QT;
      int lastkt = -1;
      for (int k0 = 0; k0 <= qt; k0 += 32) {
        const int kt = k0 + lane;
        const uint32_t bal = __ballot_sync(0xffffffffu, kt <= qt && __ldg(arow + kt) != 0);
        if (bal) lastkt = k0 + 31 - __clz(bal);
      }
      // a query tile that selects nothing still runs one (fully masked) tile, so that
      // its rows get O = 0 and LSE = -inf
      const bool none = lastkt < 0;
      if (none) lastkt = qt;
      bool first = true;
      for (int k0 = 0; ok && k0 <= qt; k0 += 32) {
        const int kl = k0 + lane;
        uint32_t bal = __ballot_sync(
            0xffffffffu, kl <= qt && (none ? kl == qt : __ldg(arow + kl) != 0));
        while (bal != 0u) {
          const int kt = k0 + __ffs(bal) - 1;
          bal &= bal - 1u;
          const int st = g % kStages;
          int go = 1;
          if (lane == 0) {
            go = mbar_wait(&tail->kv_empty[st], ((g / kStages) & 1) ^ 1u, abort_flag, p.err,
                           kErrD) ? 1 : 0;
            if (go) {
              DenseHdr& hd = tail->hdr[st];
              hd.b = b;
              hd.h = h;
              hd.qt = qt;
              hd.kt = kt;
              hd.first = first ? 1 : 0;
              hd.last = kt == lastkt ? 1 : 0;
              // the arrive releases the header; the copies complete the phase
              mbar_arrive_expect_tx(&tail->kv_full[st], L::kStage);
              const int krow = b * S + kt * kTile;
              const int kvh = h / (p.H / p.Hkv);   // the K / V head of query head h
              uint8_t* stage = smem + st * L::kStage;
#pragma unroll
              for (int a = 0; a < L::KA; ++a)
                tma_load_3d(stage + a * L::kAtom, &tm_k, &tail->kv_full[st], a * 64, kvh, krow);
#pragma unroll
              for (int a = 0; a < L::VA; ++a)
                tma_load_3d(stage + (L::KA + a) * L::kAtom, &tm_v, &tail->kv_full[st], a * 64,
                            kvh, krow);
              issued[st] = true;
              last_par[st] = (g / kStages) & 1;
            }
          }
          if (__shfl_sync(0xffffffffu, go, 0) == 0) {
            ok = false;
            break;
          }
          first = false;
          ++g;
        }
      }
    }
    // let every copy this warp started land before the CTA exits
    if (lane == 0)
      for (int st = 0; st < kStages; ++st)
        if (issued[st]) drain_wait_d(&tail->kv_full[st], last_par[st], p.err);
  } else if (warp == 1) {
    // ================================================================ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16_mn(128, kTile, false);
      constexpr uint32_t idesc_pv = umma_idesc_bf16_mn(128, DV, true);
      int g = 0;
      uint32_t qt_par = 0, of_par = 1;
      int pend = -1, pend_first = 0;   // chunk whose PV is still to be issued
      bool ok = true;
      auto issue_pv = [&](int pc, int pfirst) -> bool {
        const int pb = pc % kStages;
        if (!mbar_wait(&tail->p_full[pb], (pc / kStages) & 1, abort_flag, p.err, kErrD))
          return false;
        if (pfirst) {   // the previous item's O has been read out
          if (!mbar_wait(&tail->o_free, of_par, abort_flag, p.err, kErrD)) return false;
          of_par ^= 1u;
        }
        tc_fence_after();
        const uint32_t vbase = smem_u32(smem + pb * L::kStage + L::KA * L::kAtom);
#pragma unroll
        for (int ks = 0; ks < kTile / 16; ++ks) {
          const uint64_t bdesc = umma_sdesc_lbo(vbase + ks * 2048, L::kAtom, 1024, kLayoutSw128);
          umma_bf16_ts(tmem + L::kColO, tmem + L::kColS + pb * kTile + ks * 8, bdesc, idesc_pv,
                       (pfirst && ks == 0) ? 0u : 1u);
        }
        umma_commit(&tail->kv_empty[pb]);
        umma_commit(&tail->s_empty[pb]);
        return true;
      };
      for (int i = blockIdx.x; ok && i < nitems; i += gridDim.x) {
        bool last = false;
        while (ok && !last) {
          const int sb = g % kStages;
          const uint32_t use_par = (g / kStages) & 1;
          if (!mbar_wait(&tail->kv_full[sb], use_par, abort_flag, p.err, kErrD)) { ok = false; break; }
          const DenseHdr& hd = tail->hdr[sb];
          last = hd.last != 0;
          const int first = hd.first;
          if (first) {
            if (!mbar_wait(&tail->q_full, qt_par, abort_flag, p.err, kErrD)) { ok = false; break; }
            qt_par ^= 1u;
          }
          if (!mbar_wait(&tail->s_empty[sb], use_par ^ 1u, abort_flag, p.err, kErrD)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kbase = smem_u32(smem + sb * L::kStage);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint64_t bdesc =
                umma_sdesc(kbase + (kk >> 2) * L::kAtom + (kk & 3) * 32, 1024, kLayoutSw128);
            umma_bf16_ts(tmem + L::kColS + sb * kTile, tmem + L::kColQ + kk * 8, bdesc, idesc_s,
                         kk > 0 ? 1u : 0u);
          }
          umma_commit(&tail->s_full[sb]);
          if (pend >= 0 && !issue_pv(pend, pend_first)) { ok = false; break; }
          if (last) {
            // the item's last tile: its PV right away, so that the item's O is complete
            // before the next item's first tile arrives
            if (!issue_pv(g, first)) { ok = false; break; }
            pend = -1;
          } else {
            pend = g;
            pend_first = first;
          }
          ++g;
        }
      }
      if (ok && pend >= 0) issue_pv(pend, pend_first);
      umma_commit(&tail->drain);
      drain_wait_d(&tail->drain, 0, p.err);
    }
  } else {
    // ================================================================ softmax / output
    // warp 2 + q' + 4 * half: TMEM lane quarter (warp & 3), keys 64 * half.. of every
    // tile, Q / O columns of that half; the two warps of a quarter share each tile's
    // row max (and at the end the row sum) through shared memory
    const int quarter = warp & 3;
    const int half = (warp - kSoftWarp0) >> 2;
    const int r = quarter * 32 + lane;                     // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.scale_log2;
    // the pair's exchanges go through an mbarrier with a bounded wait, so that a
    // failure elsewhere ends both warps instead of leaving one in a barrier
    uint32_t nx = 0;
    auto pair_sync = [&]() -> bool {
      mbar_arrive(&tail->pairbar[quarter]);
      const bool r = mbar_wait(&tail->pairbar[quarter], nx & 1u, abort_flag, p.err, kErrD);
      ++nx;
      return __all_sync(0xffffffffu, r);
    };
    int g = 0;
    bool ok = true;

    // this half of the Q row (b, t = qt*128 + r, head h) -> TMEM as packed bf16 pairs;
    // rows past S load zeros and store nothing
    auto load_q = [&](int i) {
      int b, h, qt;
      item_of(i, B, H, QT, b, h, qt);
      const int t = qt * kTile + r;
      const bool in = t < S;
      const long long qrow = (static_cast<long long>(b) * S + (in ? t : 0)) * H + h;
      const uint4* src = reinterpret_cast<const uint4*>(p.Q + qrow * DQK) + half * (DQK / 16);
#pragma unroll
      for (int c = 0; c < DQK / 64; ++c) {
        uint32_t v[16];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint4 x = in ? __ldg(src + c * 4 + cc) : make_uint4(0, 0, 0, 0);
          v[cc * 4 + 0] = x.x; v[cc * 4 + 1] = x.y; v[cc * 4 + 2] = x.z; v[cc * 4 + 3] = x.w;
        }
        tmem_st_x16(tmem + lane_off + L::kColQ + half * (DQK / 4) + c * 16, v);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&tail->q_full);
    };

    if (static_cast<int>(blockIdx.x) < nitems) load_q(blockIdx.x);
    for (int i = blockIdx.x; ok && i < nitems; i += gridDim.x) {
      int b, h, qt;
      item_of(i, B, H, QT, b, h, qt);
      const int t = qt * kTile + r;
      const bool in = t < S;
      const uint32_t* brow = dp.bits + (static_cast<long long>(b) * S + (in ? t : 0)) * dp.W4;
      float m = -INFINITY, l = 0.f;   // running max (raw logits) and this half's sum
      bool last = false;
      while (!last) {
        const int sb = g % kStages;
        const uint32_t use_par = (g / kStages) & 1;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tail->s_full[sb], use_par, abort_flag, p.err, kErrD))) {
          ok = false;
          break;
        }
        // acquire the producer's header (this phase cannot advance before this tile's
        // P has been consumed)
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tail->kv_full[sb], use_par, abort_flag, p.err, kErrD))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const DenseHdr& hd = tail->hdr[sb];
        last = hd.last != 0;
        const bool first = hd.first != 0;
        const uint2 mw = in ? __ldg(reinterpret_cast<const uint2*>(brow + hd.kt * 4 + half * 2))
                            : make_uint2(0u, 0u);
        const uint32_t sbase = tmem + lane_off + L::kColS + sb * kTile;
        uint32_t sv0[32], sv1[32];
        tmem_ld_x32(sbase + half * 64, sv0);
        tmem_ld_x32(sbase + half * 64 + 32, sv1);
        tmem_ld_wait();
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if ((mw.x >> j) & 1u) mx = fmaxf(mx, __uint_as_float(sv0[j]));
          if ((mw.y >> j) & 1u) mx = fmaxf(mx, __uint_as_float(sv1[j]));
        }
        // both halves' S are in registers after this barrier, so P may overwrite them
        tail->xmax[g & 1][half][r] = mx;
        if (!pair_sync()) {
          ok = false;
          break;
        }
        mx = fmaxf(mx, tail->xmax[g & 1][half ^ 1][r]);
        if (first) {
          m = mx;
        } else if (__any_sync(0xffffffffu,
                              mx > m && (m == -INFINITY || (mx - m) * c2 > kRescaleLog2D))) {
          // refresh the running max of every row of the warp (a no-op where it has not
          // grown; the other warp of the quarter decides the same): rescale this half of
          // O (every earlier PV product is done) and l
          const int pg = g - 1;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&tail->s_empty[pg % kStages], (pg / kStages) & 1, abort_flag,
                                    p.err, kErrD))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float mnew = fmaxf(m, mx);
          const float f = m == -INFINITY ? 0.f : exp2f((m - mnew) * c2);
#pragma unroll
          for (int d0 = 0; d0 < DV / 2; d0 += 16) {
            uint32_t ov[16];
            tmem_ld_x16d(tmem + lane_off + L::kColO + half * (DV / 2) + d0, ov);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * f);
            tmem_st_x16(tmem + lane_off + L::kColO + half * (DV / 2) + d0, ov);
          }
          tmem_st_wait();
          l *= f;
          m = mnew;
        }
        // P = exp2(S*c2 - m*c2) on the selected keys, 0 elsewhere -> bf16 pairs: keys
        // 64*half.. go to columns 32*half.. of the buffer
        const float base = m == -INFINITY ? 0.f : m * c2;
        float ls = 0.f;
#pragma unroll
        for (int part = 0; part < 2; ++part) {
          const uint32_t* sv = part == 0 ? sv0 : sv1;
          const uint32_t mwp = part == 0 ? mw.x : mw.y;
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float e0 = ex2d(fmaf(__uint_as_float(sv[j]), c2, -base));
            float e1 = ex2d(fmaf(__uint_as_float(sv[j + 1]), c2, -base));
            e0 = ((mwp >> j) & 1u) ? e0 : 0.f;
            e1 = ((mwp >> (j + 1)) & 1u) ? e1 : 0.f;
            ls += e0 + e1;
            pk[j >> 1] = pack_bf16(e0, e1);
          }
          tmem_st_x16(sbase + half * 32 + part * 16, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&tail->p_full[sb]);
        l += ls;
        if (last && i + static_cast<int>(gridDim.x) < nitems) {
          // every S of this item is done: the next item's Q may replace it in TMEM
          load_q(i + gridDim.x);
        }
        ++g;
      }
      if (!ok) break;
      // final O: wait for this item's last PV, normalise, store; then release O
      const int pg = g - 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&tail->s_empty[pg % kStages], (pg / kStages) & 1,
                                              abort_flag, p.err, kErrD))) {
        ok = false;
        break;
      }
      tc_fence_after();
      tail->xl[half][r] = l;
      if (!pair_sync()) {
        ok = false;
        break;
      }
      const float lt = l + tail->xl[half ^ 1][r];
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      uint4* orow = reinterpret_cast<uint4*>(
          p.O + ((static_cast<long long>(b) * S + (in ? t : 0)) * H + h) * DV + half * (DV / 2));
#pragma unroll
      for (int d0 = 0; d0 < DV / 2; d0 += 32) {
        uint32_t ov[32];
        tmem_ld_x32(tmem + lane_off + L::kColO + half * (DV / 2) + d0, ov);
        tmem_ld_wait();
        if (in) {
#pragma unroll
          for (int d = 0; d < 32; d += 8) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(ov[d]) * inv, __uint_as_float(ov[d + 1]) * inv);
            w.y = pack_bf16(__uint_as_float(ov[d + 2]) * inv, __uint_as_float(ov[d + 3]) * inv);
            w.z = pack_bf16(__uint_as_float(ov[d + 4]) * inv, __uint_as_float(ov[d + 5]) * inv);
            w.w = pack_bf16(__uint_as_float(ov[d + 6]) * inv, __uint_as_float(ov[d + 7]) * inv);
            orow[(d0 + d) / 8] = w;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tail->o_free);
      if (in && half == 0)
        p.lse[(static_cast<long long>(b) * S + t) * H + h] =
            lt > 0.f ? (m * c2 + log2f(lt)) * 0.69314718055994530942f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

typedef CUresult (*EncodeTiledFnDense)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                       const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                       const cuuint32_t*, CUtensorMapInterleave,
                                       CUtensorMapSwizzle, CUtensorMapL2promotion,
                                       CUtensorMapFloatOOBfill);

// [rows, Hkv, cols] bf16 as (column, K/V head, row): a box of 64 columns x 1 head x 128
// rows, 128-byte swizzle (the same shared-memory tile as a [128 x 64] 2-D box); rows past
// the end read as zeros
bool make_tile_map(CUtensorMap* map, const void* base, long long rows, int Hkv, int cols) {
  static EncodeTiledFnDense fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFnDense>(ptr);
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                           static_cast<cuuint64_t>(cols) * 2 * static_cast<cuuint64_t>(Hkv)};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kTile)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DQK, int DV>
int launch_dense(const AttnParams& p, cudaStream_t stream) {
  using L = DenseLayout<DQK, DV>;
  const int QT = (p.S + kTile - 1) / kTile;
  const int W4 = QT * 4;
  // the bitmap and the tile flags live in the caller's workspace (dense_scratch_layout)
  if (p.scratch == nullptr) return DSA_ERR_WORKSPACE;
  const DenseScratch ly = dense_scratch_layout(p.B, p.S, p.H, p.Hkv, DQK, DV, false);
  uint32_t* bits = reinterpret_cast<uint32_t*>(p.scratch + ly.bits_off);
  uint8_t* any = p.scratch + ly.any_off;
  const size_t any_bytes = static_cast<size_t>(p.B) * QT * QT;
  CUtensorMap mk, mv;
  const long long krows = static_cast<long long>(p.B) * p.S;
  const size_t smem = L::kTailOff + sizeof(DenseTail);
  auto kern = attn_fwd_dense_kernel<DQK, DV>;
  if (cudaMemsetAsync(any, 0, any_bytes, stream) != cudaSuccess ||
      !make_tile_map(&mk, p.K, krows, p.Hkv, DQK) || !make_tile_map(&mv, p.V, krows, p.Hkv, DV) ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  launch_dense_mask(p.idx, p.B, p.S, p.k, W4, QT, bits, any, p.err, stream);
  const long long items = static_cast<long long>(QT) * p.B * p.H;
  const int grid = static_cast<int>(items < sms ? items : sms);
  DenseParams dp;
  dp.a = p;
  dp.bits = bits;
  dp.any = any;
  dp.W4 = W4;
  dp.QT = QT;
  kern<<<grid, kThreads, smem, stream>>>(mk, mv, dp);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

void launch_dense_mask(const int32_t* idx, int B, int S, int k, int W4, int QT, uint32_t* bits,
                       uint8_t* any, int* err, cudaStream_t stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long rows = static_cast<long long>(B) * S;
  const int grid = static_cast<int>(rows < 8LL * sms ? rows : 8LL * sms);
  dense_mask_kernel<<<grid, 256, static_cast<size_t>(W4) * 4, stream>>>(idx, B, S, k, W4, QT, bits,
                                                                       any, err);
}

// (Dqk, Dv) = (192, 128) or (128, 128), a positive scale, any Hkv dividing H (each tile is
// one head's product, so per-head K / V only changes which rows its tiles load); the
// bitmap holds B*S*ceil(S/128)*16 bytes, so S is limited to 65536.
bool attn_fwd_dense_supported(int B, int S, int H, int Dqk, int Dv, float scale) {
  const long long items = static_cast<long long>((S + kTile - 1) / kTile) * B * H;
  return scale > 0.f && S >= 1 && S <= 65536 && H >= 1 && items < (1LL << 31) &&
         ((Dqk == 192 && Dv == 128) || (Dqk == 128 && Dv == 128));
}

// The dense-tile kernel does about H * (causal 128 x 128 tiles) tile products; the
// gathered-key kernel about one 96-key chunk per row and 96 selected keys. Measured on
// GB300, a tile product costs about 5/3 of a chunk (15 against 9 ns of whole-GPU time).
// Choose the dense kernel when it is the cheaper by that count and has enough work
// items (batch x head x query tile) to give every SM one: below that its per-tile
// pipeline latency and the bitmap set-up are not hidden.
bool attn_fwd_dense_preferred(int B, int S, int H, int k) {
  const long long QT = (S + kTile - 1) / kTile;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (QT * B * H < sms) return false;
  const long long dense_units = static_cast<long long>(H) * QT * (QT + 1) / 2;
  // sum over rows t of ceil(min(t + 1, k) / 96)
  const long long N = S < k ? S : k, q = N / 96, rem = N % 96;
  const long long chunks = 96 * q * (q + 1) / 2 + rem * (q + 1) + (S - N) * ((k + 95) / 96);
  (void)B;
  return 5 * dense_units < 3 * chunks;
}

int launch_attn_fwd_dense(const AttnParams& p, int Dqk, int Dv, cudaStream_t stream) {
  if (Dqk == 192 && Dv == 128) return launch_dense<192, 128>(p, stream);
  if (Dqk == 128 && Dv == 128) return launch_dense<128, 128>(p, stream);
  return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
