// Sparse attention backward on dense tiles with a selection bitmap, for few heads
// and many selected keys per query.
//
// ("Support Ring Attention with DeepSeek DSA Sparse Indexer", Backward Flow step 6:
// dQ = dP K, dK = dP^T Q, dV = P^T dO over the same mask, "dP" read as the gradient
// of the logits; the pages evaluate it on dense blocks with partial mask blocks and
// a key-major pass for dK / dV.)
//
// The selection is the forward's bitmap (launch_dense_mask): bit s of row t is set
// when row t lists key s. P is recomputed from the forward's LSE, dS = P (dP - Delta)
// with Delta = sum_c dO O. Two kernels, because TMEM cannot hold dQ, dK, dV and the
// S / dP tiles of Dqk = 192 at once:
//
// dq kernel: item = (batch b, head h, 128 query rows); each TMEM lane is a query row.
//   Per 64-key half of every active 128-key tile (K / V tiles by TMA, 2-stage ring):
//     S  = Q . K^T    (A = Q in TMEM, B = K rows in smem, K-major)        N = 64
//     dP = dO . V^T   (A = dO in TMEM, B = V rows, K-major)               N = 64
//     dS -> bf16 tile in smem (double-buffered)
//     dQ += dS . K    (A = dS in smem, B = K rows MN-major)               N = Dqk
//   dQ stays in TMEM for the item and is written once (bf16, times scale). The
//   kernel also writes Delta for the dk/dv kernel.
//   TMEM: [Q: Dqk/2][dO: Dv/2][S: 64][dP: 64][dQ: Dqk].
//
// dk/dv kernel: item = (batch b, 128-key tile, group of heads); each TMEM lane is a key.
//   K / V of the tile stay in smem for the item; per head of the group and per 64-query
//   half of every active query tile (Q / dO rows by TMA, 2-stage ring, with the rows'
//   LSE, Delta and bitmap words staged beside them):
//     S^T  = K . Q^T   (A = K tile, B = Q rows, both K-major)             N = 64
//     dP^T = V . dO^T  (A = V tile, B = dO rows)                          N = 64
//     P^T, dS^T -> bf16 pairs in TMEM over the S^T / dP^T columns already read
//     dV += P^T . dO   (A = P^T in TMEM, B = dO rows MN-major)            N = Dv
//     dK += dS^T . Q   (A = dS^T in TMEM, B = Q rows MN-major)            N = Dqk
//   At the end of an item each lane adds its key's dK (times scale) and dV rows into
//   the fp32 [B*S, Dqk+Dv] workspace with 16-byte reductions (groups of heads add
//   into the same rows), which finalize_dkv converts to bf16.
//   TMEM: [dK: Dqk][dV: Dv][S^T: 64][dP^T: 64].
//
// Both: warp 0 TMA producer, warp 1 TMEM owner and UMMA issuer, warps 2-5 softmax /
// epilogue (TMEM lane quarters 2, 3, 0, 1); persistent, heaviest items first; every
// wait is bounded (2 s), after which the kernel reports DSA_STAGE_BWD | TIMEOUT.

#include "dsa_attn_common.cuh"

namespace dsa {
namespace {

constexpr int kT = 128;               // rows of a query or key tile
constexpr int kH = 64;                // keys (dq) or queries (dk/dv) per half step
constexpr int kThreadsB = 192;
constexpr int kErrB2 = DSA_STAGE_BWD | DSA_DEVERR_TIMEOUT;
constexpr int kGroupHeads = 1;        // heads per dk/dv item (1, 2, 4 measured: 1 is fastest)
// every head of an item reads one K / V head (with per-head K / V only single-head items do)
static_assert(kGroupHeads == 1, "an item's heads must share one K / V head");

struct DenseBwdParams {
  AttnParams a;
  const uint32_t* bits;   // [B*S, W4]
  const uint8_t* any;     // [B, QT, QT]
  float* delta;           // [B*S*H]: written by the dq kernel, read by the dk/dv kernel
  int W4, QT;
};

struct BwdHdr {
  int b, h, qt, kt;
  int first, last;
  int pad[2];
};

__device__ __forceinline__ void bwd_drain_wait(uint64_t* bar, uint32_t parity, int* err) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report_error(err, kErrB2);
      return;
    }
  }
}

__device__ __forceinline__ float ex2bd(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_ld_x16e(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

// ============================================================================ dq kernel

template <int DQK, int DV>
struct DqLayout {
  static constexpr int KA = DQK / 64, VA = DV / 64;
  static constexpr uint32_t kAtom = kT * 128;                 // [128 key rows x 128 B]
  static constexpr uint32_t kStage = (KA + VA) * kAtom;
  static constexpr uint32_t kDsOff = 2 * kStage;              // 2 dS tiles [128 q x 64 keys]
  static constexpr uint32_t kDsTile = kT * 128;
  static constexpr uint32_t kTailOff = kDsOff + 2 * kDsTile;
  static constexpr uint32_t kColQ = 0, kColDO = DQK / 2, kColS = kColDO + DV / 2,
                            kColDP = kColS + kH, kColDQ = kColDP + kH;
  static_assert(kColDQ + DQK <= 512, "TMEM budget");
};

struct DqTail {
  BwdHdr hdr[2];
  uint64_t kv_full[2], kv_empty[2];
  uint64_t sdp_full, sdp_free;
  uint64_t ds_full[2], ds_free[2];
  uint64_t qdo_full, dq_full, dq_free;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

__device__ __forceinline__ void dq_item(int i, int B, int H, int QT, int& b, int& h, int& qt) {
  const int bh = B * H;
  qt = QT - 1 - i / bh;
  const int r = i - (QT - 1 - qt) * bh;
  b = r / H;
  h = r - b * H;
}

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreadsB, 1)
    attn_bwd_dense_dq_kernel(const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const DenseBwdParams dp) {
  using L = DqLayout<DQK, DV>;
  const AttnParams& p = dp.a;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) report_error(p.err, DSA_STAGE_BWD | DSA_DEVERR_MISALIGNED);
    return;
  }
  DqTail* tail = reinterpret_cast<DqTail*>(smem + L::kTailOff);
  volatile int* abort_flag = &tail->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.B, S = p.S, H = p.H, QT = dp.QT;
  const int nitems = QT * B * H;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tail->kv_full[i], 1);
      mbar_init(&tail->kv_empty[i], 1);
      mbar_init(&tail->ds_full[i], 128);
      mbar_init(&tail->ds_free[i], 1);
    }
    mbar_init(&tail->sdp_full, 1);
    mbar_init(&tail->sdp_free, 128);
    mbar_init(&tail->qdo_full, 128);
    mbar_init(&tail->dq_full, 1);
    mbar_init(&tail->dq_free, 128);
    mbar_init(&tail->drain, 1);
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
    int g = 0;
    bool ok = true;
    uint32_t last_par[2] = {0, 0};
    bool issued[2] = {false, false};
    for (int i = blockIdx.x; ok && i < nitems; i += gridDim.x) {
      int b, h, qt;
      dq_item(i, B, H, QT, b, h, qt);
      const uint8_t* arow = dp.any + (static_cast<long long>(b) * QT + qt) * QT;
      int lastkt = -1;
      for (int k0 = 0; k0 <= qt; k0 += 32) {
        const int kt = k0 + lane;
        const uint32_t bal = __ballot_sync(0xffffffffu, kt <= qt && __ldg(arow + kt) != 0);
        if (bal) lastkt = k0 + 31 - __clz(bal);
      }
      const bool none = lastkt < 0;   // still one (fully masked) tile: dQ = 0
      if (none) lastkt = qt;
      bool first = true;
      for (int k0 = 0; ok && k0 <= qt; k0 += 32) {
        const int kl = k0 + lane;
        uint32_t bal = __ballot_sync(
            0xffffffffu, kl <= qt && (none ? kl == qt : __ldg(arow + kl) != 0));
        while (bal != 0u) {
          const int kt = k0 + __ffs(bal) - 1;
          bal &= bal - 1u;
          const int st = g & 1;
          int go = 1;
          if (lane == 0) {
            go = mbar_wait(&tail->kv_empty[st], ((g >> 1) & 1) ^ 1u, abort_flag, p.err, kErrB2)
                     ? 1 : 0;
            if (go) {
              BwdHdr& hd = tail->hdr[st];
              hd.b = b;
              hd.h = h;
              hd.qt = qt;
              hd.kt = kt;
              hd.first = first ? 1 : 0;
              hd.last = kt == lastkt ? 1 : 0;
              mbar_arrive_expect_tx(&tail->kv_full[st], L::kStage);
              const int krow = b * S + kt * kT;
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
              last_par[st] = (g >> 1) & 1;
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
    if (lane == 0)
      for (int st = 0; st < 2; ++st)
        if (issued[st]) bwd_drain_wait(&tail->kv_full[st], last_par[st], p.err);
  } else if (warp == 1) {
    // ================================================================ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16_mn(128, kH, false);
      constexpr uint32_t idesc_dq = umma_idesc_bf16_mn(128, DQK, true);
      const uint32_t ds0 = smem_u32(smem + L::kDsOff);
      int g = 0;
      uint32_t qd_par = 0, of_par = 1;
      bool ok = true;
      // dQ += dS(u) . K rows of half c of stage st
      auto issue_dq = [&](int u, int st, int c, bool first_sub, bool last_sub) -> bool {
        if (!mbar_wait(&tail->ds_full[u & 1], (u >> 1) & 1, abort_flag, p.err, kErrB2)) return false;
        if (first_sub) {   // the previous item's dQ has been read out
          if (!mbar_wait(&tail->dq_free, of_par, abort_flag, p.err, kErrB2)) return false;
          of_par ^= 1u;
        }
        tc_fence_after();
        const uint32_t kst = smem_u32(smem + st * L::kStage) + c * (kH * 128);
#pragma unroll
        for (int kk = 0; kk < kH / 16; ++kk)
          umma_bf16(tmem + L::kColDQ,
                    umma_sdesc(ds0 + (u & 1) * L::kDsTile + kk * 32, 1024, kLayoutSw128),
                    umma_sdesc_lbo(kst + kk * 2048, L::kAtom, 1024, kLayoutSw128), idesc_dq,
                    (first_sub && kk == 0) ? 0u : 1u);
        umma_commit(&tail->ds_free[u & 1]);
        if (c == 1) umma_commit(&tail->kv_empty[st]);   // K / V of the stage are read
        if (last_sub) umma_commit(&tail->dq_full);
        return true;
      };
      int pu = -1, pst = 0, pc = 0;
      bool pfirst = false, plast = false;
      for (int i = blockIdx.x; ok && i < nitems; i += gridDim.x) {
        bool last = false;
        while (ok && !last) {
          const int st = g & 1;
          if (!mbar_wait(&tail->kv_full[st], (g >> 1) & 1, abort_flag, p.err, kErrB2)) { ok = false; break; }
          const BwdHdr& hd = tail->hdr[st];
          last = hd.last != 0;
          const bool first = hd.first != 0;
          if (first) {
            if (!mbar_wait(&tail->qdo_full, qd_par, abort_flag, p.err, kErrB2)) { ok = false; break; }
            qd_par ^= 1u;
          }
          const uint32_t kst = smem_u32(smem + st * L::kStage);
          for (int c = 0; c < 2; ++c) {
            const int u = 2 * g + c;
            // S / dP of the previous half have been read by the softmax warps
            if (u > 0 && !mbar_wait(&tail->sdp_free, (u - 1) & 1, abort_flag, p.err, kErrB2)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t kb = kst + c * (kH * 128);
#pragma unroll
            for (int kk = 0; kk < DQK / 16; ++kk)
              umma_bf16_ts(tmem + L::kColS, tmem + L::kColQ + kk * 8,
                           umma_sdesc(kb + (kk >> 2) * L::kAtom + (kk & 3) * 32, 1024, kLayoutSw128),
                           idesc_s, kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < DV / 16; ++kk)
              umma_bf16_ts(tmem + L::kColDP, tmem + L::kColDO + kk * 8,
                           umma_sdesc(kb + (L::KA + (kk >> 2)) * L::kAtom + (kk & 3) * 32, 1024,
                                      kLayoutSw128),
                           idesc_s, kk > 0 ? 1u : 0u);
            umma_commit(&tail->sdp_full);
            // the previous half's dQ product while the softmax warps work on this one
            if (pu >= 0 && !issue_dq(pu, pst, pc, pfirst, plast)) { ok = false; break; }
            pu = u;
            pst = st;
            pc = c;
            pfirst = first && c == 0;
            plast = last && c == 1;
          }
          if (!ok) break;
          if (last) {   // the item's dQ is complete before the next item starts
            if (!issue_dq(pu, pst, pc, pfirst, plast)) { ok = false; break; }
            pu = -1;
          }
          ++g;
        }
      }
      if (ok && pu >= 0) issue_dq(pu, pst, pc, pfirst, plast);
      umma_commit(&tail->drain);
      bwd_drain_wait(&tail->drain, 0, p.err);
    }
  } else {
    // ================================================================ softmax / epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                     // query row within the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.scale_log2;
    uint8_t* dsrow0 = smem + L::kDsOff + r * 128;
    const uint32_t sw = static_cast<uint32_t>(r & 7);
    float nx_delta = 0.f, nx_lse2 = 0.f;

    // Q and dO rows of (b, t = qt*128 + r, head h) -> TMEM (packed bf16 pairs), and the
    // row's Delta = sum_c dO O and LSE * log2(e); rows past S load zeros
    auto load_qdo = [&](int i) {
      int b, h, qt;
      dq_item(i, B, H, QT, b, h, qt);
      const int t = qt * kT + r;
      const bool in = t < S;
      const long long qrow = (static_cast<long long>(b) * S + (in ? t : 0)) * H + h;
      const uint4* q4 = reinterpret_cast<const uint4*>(p.Q + qrow * DQK);
      const uint4* d4 = reinterpret_cast<const uint4*>(p.dO + qrow * DV);
      const uint4* o4 = reinterpret_cast<const uint4*>(p.O_in + qrow * DV);
#pragma unroll
      for (int c = 0; c < DQK / 32; ++c) {
        uint32_t v[16];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint4 x = in ? __ldg(q4 + c * 4 + cc) : make_uint4(0, 0, 0, 0);
          v[cc * 4 + 0] = x.x; v[cc * 4 + 1] = x.y; v[cc * 4 + 2] = x.z; v[cc * 4 + 3] = x.w;
        }
        tmem_st_x16(tmem + lane_off + L::kColQ + c * 16, v);
      }
      float delta = 0.f;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t v[16];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint4 x = in ? __ldg(d4 + c * 4 + cc) : make_uint4(0, 0, 0, 0);
          const uint4 o = in ? __ldg(o4 + c * 4 + cc) : make_uint4(0, 0, 0, 0);
          v[cc * 4 + 0] = x.x; v[cc * 4 + 1] = x.y; v[cc * 4 + 2] = x.z; v[cc * 4 + 3] = x.w;
          const uint32_t xv[4] = {x.x, x.y, x.z, x.w}, ov[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            delta = fmaf(__uint_as_float(xv[e] << 16), __uint_as_float(ov[e] << 16), delta);
            delta = fmaf(__uint_as_float(xv[e] & 0xffff0000u), __uint_as_float(ov[e] & 0xffff0000u),
                         delta);
          }
        }
        tmem_st_x16(tmem + lane_off + L::kColDO + c * 16, v);
      }
      nx_delta = delta;
      nx_lse2 = in ? p.lse_in[qrow] * 1.4426950408889634f : 0.f;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&tail->qdo_full);
    };

    int g = 0;
    uint32_t dq_par = 0;
    bool ok = true;
    if (static_cast<int>(blockIdx.x) < nitems) load_qdo(blockIdx.x);
    for (int i = blockIdx.x; ok && i < nitems; i += gridDim.x) {
      int b, h, qt;
      dq_item(i, B, H, QT, b, h, qt);
      const int t = qt * kT + r;
      const bool in = t < S;
      const long long qrow = (static_cast<long long>(b) * S + (in ? t : 0)) * H + h;
      const uint32_t* brow = dp.bits + (static_cast<long long>(b) * S + (in ? t : 0)) * dp.W4;
      const float delta = nx_delta, lse2 = nx_lse2;
      bool last = false;
      while (ok && !last) {
        const int st = g & 1;
        int kt = 0;
        for (int c = 0; c < 2; ++c) {
          const int u = 2 * g + c;
          if (!__all_sync(0xffffffffu, mbar_wait(&tail->sdp_full, u & 1, abort_flag, p.err, kErrB2))) {
            ok = false;
            break;
          }
          if (c == 0) {
            // the producer's header (this phase cannot advance before this tile's dQ
            // products have read the stage)
            if (!__all_sync(0xffffffffu, mbar_wait(&tail->kv_full[st], (g >> 1) & 1, abort_flag,
                                                    p.err, kErrB2))) {
              ok = false;
              break;
            }
            kt = tail->hdr[st].kt;
            last = tail->hdr[st].last != 0;
          }
          tc_fence_after();
          const uint2 mw = in ? __ldg(reinterpret_cast<const uint2*>(brow + kt * 4 + 2 * c))
                              : make_uint2(0u, 0u);
          uint32_t dw[32];
#pragma unroll
          for (int qk = 0; qk < 4; ++qk) {
            uint32_t sv[16], dv[16];
            tmem_ld_x16e(tmem + lane_off + L::kColS + qk * 16, sv);
            tmem_ld_x16e(tmem + lane_off + L::kColDP + qk * 16, dv);
            tmem_ld_wait();
            const uint32_t vm = (qk < 2 ? mw.x : mw.y) >> ((qk & 1) * 16);
#pragma unroll
            for (int j = 0; j < 16; j += 2) {
              const float p0 = ((vm >> j) & 1u) ? ex2bd(fmaf(__uint_as_float(sv[j]), c2, -lse2)) : 0.f;
              const float p1 =
                  ((vm >> (j + 1)) & 1u) ? ex2bd(fmaf(__uint_as_float(sv[j + 1]), c2, -lse2)) : 0.f;
              dw[qk * 8 + j / 2] = pack_bf16(p0 * (__uint_as_float(dv[j]) - delta),
                                             p1 * (__uint_as_float(dv[j + 1]) - delta));
            }
          }
          tc_fence_before();
          mbar_arrive(&tail->sdp_free);
          // dS into its buffer once the product two halves back has read it
          if (u >= 2 && !__all_sync(0xffffffffu, mbar_wait(&tail->ds_free[u & 1], ((u >> 1) - 1) & 1,
                                                           abort_flag, p.err, kErrB2))) {
            ok = false;
            break;
          }
          uint8_t* dsrow = dsrow0 + (u & 1) * L::kDsTile;
#pragma unroll
          for (int cc = 0; cc < 8; ++cc) {
            const uint32_t off = (static_cast<uint32_t>(cc) ^ sw) << 4;
            *reinterpret_cast<uint4*>(dsrow + off) =
                make_uint4(dw[cc * 4], dw[cc * 4 + 1], dw[cc * 4 + 2], dw[cc * 4 + 3]);
          }
          fence_proxy_async_smem();
          tc_fence_before();
          mbar_arrive(&tail->ds_full[u & 1]);
          if (last && c == 1 && i + static_cast<int>(gridDim.x) < nitems) {
            // every S / dP of this item is done: the next item's Q / dO may replace them
            load_qdo(i + gridDim.x);
          }
        }
        ++g;
      }
      if (!ok) break;
      // dQ of the item (times scale), then release the accumulator; Delta for dK / dV
      if (!__all_sync(0xffffffffu, mbar_wait(&tail->dq_full, dq_par, abort_flag, p.err, kErrB2))) {
        ok = false;
        break;
      }
      dq_par ^= 1u;
      tc_fence_after();
      uint4* qd = reinterpret_cast<uint4*>(p.dQ + qrow * DQK);
#pragma unroll
      for (int d0 = 0; d0 < DQK; d0 += 32) {
        uint32_t v[32];
        tmem_ld_x32(tmem + lane_off + L::kColDQ + d0, v);
        tmem_ld_wait();
        if (in) {
#pragma unroll
          for (int d = 0; d < 32; d += 8) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(v[d]) * p.scale, __uint_as_float(v[d + 1]) * p.scale);
            w.y = pack_bf16(__uint_as_float(v[d + 2]) * p.scale, __uint_as_float(v[d + 3]) * p.scale);
            w.z = pack_bf16(__uint_as_float(v[d + 4]) * p.scale, __uint_as_float(v[d + 5]) * p.scale);
            w.w = pack_bf16(__uint_as_float(v[d + 6]) * p.scale, __uint_as_float(v[d + 7]) * p.scale);
            qd[(d0 + d) / 8] = w;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tail->dq_free);
      if (in) dp.delta[qrow] = delta;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ========================================================================= dk/dv kernel

template <int DQK, int DV>
struct DkvLayout {
  static constexpr int KA = DQK / 64, VA = DV / 64;
  static constexpr uint32_t kKvAtom = kT * 128;               // [128 key rows x 128 B]
  static constexpr uint32_t kKv = (KA + VA) * kKvAtom;        // the item's K / V tile
  static constexpr uint32_t kQAtom = kH * 128;                // [64 query rows x 128 B]
  static constexpr uint32_t kRows = (KA + VA) * kQAtom;       // Q and dO rows of a step
  static constexpr uint32_t kInfo = kRows;                    // then lse2[64], delta[64], words[64][4]
  static constexpr uint32_t kStage = (kRows + 2 * kH * 4 + kH * 16 + 1023) / 1024 * 1024;
  static constexpr uint32_t kStageOff = kKv;
  static constexpr uint32_t kTailOff = kStageOff + 2 * kStage;
  static constexpr uint32_t kColDK = 0, kColDV = DQK, kColS = DQK + DV, kColDP = kColS + kH,
                            kColP = kColDP + kH, kColDS = kColP + kH / 2;
  static_assert(kColDS + kH / 2 <= 512, "TMEM budget");
};

struct DkvHdr {
  int h, q0, first, last;   // first / last step of the item
};

struct DkvTail {
  DkvHdr hdr[2];
  uint64_t kv_full, kv_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t sdp_full, sdp_free, pds_full, pds_free;
  uint64_t dkv_full, dkv_free;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};

// item i -> (key tile kt, batch b, head group hg); small kt first (the most query tiles)
__device__ __forceinline__ void dkv_item(int i, int B, int HGN, int& kt, int& b, int& hg) {
  const int per = B * HGN;
  kt = i / per;
  const int r = i - kt * per;
  b = r / HGN;
  hg = r - b * HGN;
}

// does any query tile qi >= kt of batch b select a key of tile kt (all lanes agree)
__device__ __forceinline__ bool dkv_active(const uint8_t* any, int b, int kt, int QT, int lane) {
  bool a = false;
  for (int q0 = kt; q0 < QT; q0 += 32) {
    const int qi = q0 + lane;
    a |= __any_sync(0xffffffffu, qi < QT && __ldg(any + (static_cast<long long>(b) * QT + qi) * QT + kt) != 0);
  }
  return a;
}

// the same test from a single thread
__device__ __forceinline__ bool dkv_active_1(const uint8_t* any, int b, int kt, int QT) {
  for (int qi = kt; qi < QT; ++qi)
    if (__ldg(any + (static_cast<long long>(b) * QT + qi) * QT + kt) != 0) return true;
  return false;
}

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreadsB, 1)
    attn_bwd_dense_dkv_kernel(const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v,
                              const __grid_constant__ CUtensorMap tm_q,
                              const __grid_constant__ CUtensorMap tm_do, const DenseBwdParams dp) {
  using L = DkvLayout<DQK, DV>;
  const AttnParams& p = dp.a;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) report_error(p.err, DSA_STAGE_BWD | DSA_DEVERR_MISALIGNED);
    return;
  }
  DkvTail* tail = reinterpret_cast<DkvTail*>(smem + L::kTailOff);
  volatile int* abort_flag = &tail->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = p.B, S = p.S, H = p.H, QT = dp.QT;
  const int HGN = (H + kGroupHeads - 1) / kGroupHeads;
  const int nitems = QT * B * HGN;

  if (threadIdx.x == 0) {
    mbar_init(&tail->kv_full, 1);
    mbar_init(&tail->kv_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tail->q_full[i], 33);   // lane 0's copies + 32 lanes' staged row data
      mbar_init(&tail->q_empty[i], 1);
    }
    mbar_init(&tail->sdp_full, 1);
    mbar_init(&tail->sdp_free, 128);
    mbar_init(&tail->pds_full, 128);
    mbar_init(&tail->pds_free, 1);
    mbar_init(&tail->dkv_full, 1);
    mbar_init(&tail->dkv_free, 128);
    mbar_init(&tail->drain, 1);
    tail->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
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
    // per item: the K / V tile; per step (head, 64 query rows): Q and dO rows by TMA
    // and, from the lanes, the rows' LSE * log2(e), Delta and bitmap words of the tile
    int u = 0, n = 0;
    bool ok = true;
    uint32_t q_last[2] = {0, 0};
    bool q_issued[2] = {false, false}, kv_issued = false;
    uint32_t kv_last = 0;
    for (int i = blockIdx.x; ok && i < nitems; i += gridDim.x) {
      int kt, b, hg;
      dkv_item(i, B, HGN, kt, b, hg);
      if (!dkv_active(dp.any, b, kt, QT, lane)) continue;
      int go = 1;
      if (lane == 0) {
        go = mbar_wait(&tail->kv_empty, (n & 1) ^ 1u, abort_flag, p.err, kErrB2) ? 1 : 0;
        if (go) {
          mbar_arrive_expect_tx(&tail->kv_full, L::kKv);
          const int krow = b * S + kt * kT;
          const int kvh = hg * kGroupHeads / (p.H / p.Hkv);   // the item's K / V head
#pragma unroll
          for (int a = 0; a < L::KA; ++a)
            tma_load_3d(smem + a * L::kKvAtom, &tm_k, &tail->kv_full, a * 64, kvh, krow);
#pragma unroll
          for (int a = 0; a < L::VA; ++a)
            tma_load_3d(smem + (L::KA + a) * L::kKvAtom, &tm_v, &tail->kv_full, a * 64, kvh,
                        krow);
          kv_issued = true;
          kv_last = n & 1;
        }
      }
      if (__shfl_sync(0xffffffffu, go, 0) == 0) break;
      ++n;
      const uint8_t* acol = dp.any + static_cast<long long>(b) * QT * QT + kt;
      // the last active query tile of the column (for the last-step flag)
      int lastqi = kt;
      for (int q0 = kt; q0 < QT; q0 += 32) {
        const int qi = q0 + lane;
        const uint32_t bal = __ballot_sync(0xffffffffu, qi < QT && __ldg(acol + static_cast<long long>(qi) * QT) != 0);
        if (bal) lastqi = q0 + 31 - __clz(bal);
      }
      const int h_end = min(H, (hg + 1) * kGroupHeads);
      bool first = true;
      for (int h = hg * kGroupHeads; ok && h < h_end; ++h) {
        for (int q0 = kt; ok && q0 < QT; q0 += 32) {
          const int ql = q0 + lane;
          uint32_t bal = __ballot_sync(0xffffffffu, ql < QT && __ldg(acol + static_cast<long long>(ql) * QT) != 0);
          while (bal != 0u) {
            const int qi = q0 + __ffs(bal) - 1;
            bal &= bal - 1u;
            for (int c = 0; c < 2; ++c) {
              const int st = u & 1;
              int g2 = 1;
              if (lane == 0)
                g2 = mbar_wait(&tail->q_empty[st], ((u >> 1) & 1) ^ 1u, abort_flag, p.err, kErrB2) ? 1 : 0;
              if (__shfl_sync(0xffffffffu, g2, 0) == 0) {
                ok = false;
                break;
              }
              uint8_t* stage = smem + L::kStageOff + st * L::kStage;
              const int qrow0 = qi * kT + c * kH;            // first query row of the step
              // staged row data: lanes take rows j = lane and lane + 32
              float* lse2 = reinterpret_cast<float*>(stage + L::kInfo);
              float* dlt = lse2 + kH;
              uint4* words = reinterpret_cast<uint4*>(dlt + kH);
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int j = lane + 32 * e, t = qrow0 + j;
                const bool in = t < S;
                const long long qr = (static_cast<long long>(b) * S + (in ? t : 0)) * H + h;
                lse2[j] = in ? p.lse_in[qr] * 1.4426950408889634f : 0.f;
                dlt[j] = in ? dp.delta[qr] : 0.f;
                words[j] = in ? __ldg(reinterpret_cast<const uint4*>(
                                    dp.bits + (static_cast<long long>(b) * S + t) * dp.W4 + kt * 4))
                              : make_uint4(0u, 0u, 0u, 0u);
              }
              if (lane == 0) {
                DkvHdr& hd = tail->hdr[st];
                hd.h = h;
                hd.q0 = qrow0;
                hd.first = first ? 1 : 0;
                hd.last = (h == h_end - 1 && qi == lastqi && c == 1) ? 1 : 0;
                mbar_arrive_expect_tx(&tail->q_full[st], L::kRows);
                const int row = b * S + qrow0;
#pragma unroll
                for (int a = 0; a < L::KA; ++a)
                  tma_load_3d(stage + a * L::kQAtom, &tm_q, &tail->q_full[st], a * 64, h, row);
#pragma unroll
                for (int a = 0; a < L::VA; ++a)
                  tma_load_3d(stage + (L::KA + a) * L::kQAtom, &tm_do, &tail->q_full[st], a * 64, h,
                              row);
                q_issued[st] = true;
                q_last[st] = (u >> 1) & 1;
              }
              mbar_arrive(&tail->q_full[st]);   // each lane releases its staged row data
              first = false;
              ++u;
            }
            if (!ok) break;
          }
        }
      }
    }
    if (lane == 0) {
      if (kv_issued) bwd_drain_wait(&tail->kv_full, kv_last, p.err);
      for (int st = 0; st < 2; ++st)
        if (q_issued[st]) bwd_drain_wait(&tail->q_full[st], q_last[st], p.err);
    }
  } else if (warp == 1) {
    // ================================================================ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_st = umma_idesc_bf16_mn(128, kH, false);
      constexpr uint32_t idesc_dv = umma_idesc_bf16_mn(128, DV, true);
      constexpr uint32_t idesc_dk = umma_idesc_bf16_mn(128, DQK, true);
      const uint32_t kv = smem_u32(smem);
      int u = 0, n = 0;
      uint32_t fr_par = 1;
      bool ok = true;
      // dV += P^T . dO and dK += dS^T . Q of step pu, once its P^T / dS^T are in TMEM
      auto issue_grads = [&](int pu, bool pfirst, bool plast) -> bool {
        if (!mbar_wait(&tail->pds_full, pu & 1, abort_flag, p.err, kErrB2)) return false;
        if (pfirst) {   // the previous item's dK / dV have been read out
          if (!mbar_wait(&tail->dkv_free, fr_par, abort_flag, p.err, kErrB2)) return false;
          fr_par ^= 1u;
        }
        tc_fence_after();
        const uint32_t rows = smem_u32(smem + L::kStageOff + (pu & 1) * L::kStage);
#pragma unroll
        for (int kk = 0; kk < kH / 16; ++kk)
          umma_bf16_ts(tmem + L::kColDV, tmem + L::kColP + kk * 8,
                       umma_sdesc_lbo(rows + L::KA * L::kQAtom + kk * 2048, L::kQAtom, 1024,
                                      kLayoutSw128),
                       idesc_dv, (pfirst && kk == 0) ? 0u : 1u);
#pragma unroll
        for (int kk = 0; kk < kH / 16; ++kk)
          umma_bf16_ts(tmem + L::kColDK, tmem + L::kColDS + kk * 8,
                       umma_sdesc_lbo(rows + kk * 2048, L::kQAtom, 1024, kLayoutSw128), idesc_dk,
                       (pfirst && kk == 0) ? 0u : 1u);
        umma_commit(&tail->pds_free);
        umma_commit(&tail->q_empty[pu & 1]);   // the step's Q / dO rows are read
        if (plast) umma_commit(&tail->dkv_full);
        return true;
      };
      int pu = -1;
      bool pfirst = false, plast = false;
      for (int i = blockIdx.x; ok && i < nitems; i += gridDim.x) {
        int kt, b, hg;
        dkv_item(i, B, HGN, kt, b, hg);
        if (!dkv_active_1(dp.any, b, kt, QT)) continue;
        if (!mbar_wait(&tail->kv_full, n & 1, abort_flag, p.err, kErrB2)) break;
        ++n;
        bool last = false;
        while (ok && !last) {
          const int st = u & 1;
          if (!mbar_wait(&tail->q_full[st], (u >> 1) & 1, abort_flag, p.err, kErrB2)) { ok = false; break; }
          const DkvHdr& hd = tail->hdr[st];
          last = hd.last != 0;
          const bool first = hd.first != 0;
          // S^T / dP^T of the previous step have been read by the softmax warps
          if (u > 0 && !mbar_wait(&tail->sdp_free, (u - 1) & 1, abort_flag, p.err, kErrB2)) { ok = false; break; }
          tc_fence_after();
          const uint32_t rows = smem_u32(smem + L::kStageOff + st * L::kStage);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk)
            umma_bf16(tmem + L::kColS,
                      umma_sdesc(kv + (kk >> 2) * L::kKvAtom + (kk & 3) * 32, 1024, kLayoutSw128),
                      umma_sdesc(rows + (kk >> 2) * L::kQAtom + (kk & 3) * 32, 1024, kLayoutSw128),
                      idesc_st, kk > 0 ? 1u : 0u);
#pragma unroll
          for (int kk = 0; kk < DV / 16; ++kk)
            umma_bf16(tmem + L::kColDP,
                      umma_sdesc(kv + (L::KA + (kk >> 2)) * L::kKvAtom + (kk & 3) * 32, 1024,
                                 kLayoutSw128),
                      umma_sdesc(rows + (L::KA + (kk >> 2)) * L::kQAtom + (kk & 3) * 32, 1024,
                                 kLayoutSw128),
                      idesc_st, kk > 0 ? 1u : 0u);
          umma_commit(&tail->sdp_full);
          if (last) umma_commit(&tail->kv_empty);   // the item's K / V tile is read
          if (pu >= 0 && !issue_grads(pu, pfirst, plast)) { ok = false; break; }
          pu = u;
          pfirst = first;
          plast = last;
          if (last) {   // the item's dK / dV are complete before the next item starts
            if (!issue_grads(pu, pfirst, plast)) { ok = false; break; }
            pu = -1;
          }
          ++u;
        }
      }
      if (ok && pu >= 0) issue_grads(pu, pfirst, plast);
      umma_commit(&tail->drain);
      bwd_drain_wait(&tail->drain, 0, p.err);
    }
  } else {
    // ================================================================ softmax / epilogue
    // each lane is key s = kt*128 + r of the item's tile; bit (s & 31) = lane of word
    // r >> 5 = quarter of a query row's tile words
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.scale_log2;
    int u = 0;
    uint32_t dkv_par = 0;
    bool ok = true;
    for (int i = blockIdx.x; ok && i < nitems; i += gridDim.x) {
      int kt, b, hg;
      dkv_item(i, B, HGN, kt, b, hg);
      if (!dkv_active(dp.any, b, kt, QT, lane)) continue;
      const int s = kt * kT + r;
      const bool kin = s < S;
      bool last = false;
      while (!last) {
        const int st = u & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&tail->sdp_full, u & 1, abort_flag, p.err, kErrB2))) {
          ok = false;
          break;
        }
        // the staged row data and header (this phase cannot advance before this step's
        // dV / dK products have read the rows)
        if (!__all_sync(0xffffffffu, mbar_wait(&tail->q_full[st], (u >> 1) & 1, abort_flag, p.err,
                                                kErrB2))) {
          ok = false;
          break;
        }
        tc_fence_after();
        last = tail->hdr[st].last != 0;
        const uint8_t* stage = smem + L::kStageOff + st * L::kStage;
        const float* lse2 = reinterpret_cast<const float*>(stage + L::kInfo);
        const float* dlt = lse2 + kH;
        const uint32_t* wq = reinterpret_cast<const uint32_t*>(dlt + kH) + quarter;
        uint32_t pw[32], dw[32];
#pragma unroll
        for (int qk = 0; qk < 4; ++qk) {
          uint32_t sv[16], dv[16];
          tmem_ld_x16e(tmem + lane_off + L::kColS + qk * 16, sv);
          tmem_ld_x16e(tmem + lane_off + L::kColDP + qk * 16, dv);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const int q = qk * 16 + j;
            const bool v0 = (wq[q * 4] >> lane) & 1u, v1 = (wq[(q + 1) * 4] >> lane) & 1u;
            const float p0 = v0 ? ex2bd(fmaf(__uint_as_float(sv[j]), c2, -lse2[q])) : 0.f;
            const float p1 = v1 ? ex2bd(fmaf(__uint_as_float(sv[j + 1]), c2, -lse2[q + 1])) : 0.f;
            pw[q / 2] = pack_bf16(p0, p1);
            dw[q / 2] = pack_bf16(p0 * (__uint_as_float(dv[j]) - dlt[q]),
                                  p1 * (__uint_as_float(dv[j + 1]) - dlt[q + 1]));
          }
        }
        tc_fence_before();
        mbar_arrive(&tail->sdp_free);
        // the previous step's dV / dK products have read their P^T / dS^T
        if (u > 0 && !__all_sync(0xffffffffu, mbar_wait(&tail->pds_free, (u - 1) & 1, abort_flag,
                                                         p.err, kErrB2))) {
          ok = false;
          break;
        }
        uint32_t a16[16];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
#pragma unroll
          for (int j = 0; j < 16; ++j) a16[j] = pw[h2 * 16 + j];
          tmem_st_x16(tmem + lane_off + L::kColP + h2 * 16, a16);
#pragma unroll
          for (int j = 0; j < 16; ++j) a16[j] = dw[h2 * 16 + j];
          tmem_st_x16(tmem + lane_off + L::kColDS + h2 * 16, a16);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&tail->pds_full);
        ++u;
      }
      if (!ok) break;
      // the item's dK (times scale) and dV rows of this key into the fp32 workspace
      if (!__all_sync(0xffffffffu, mbar_wait(&tail->dkv_full, dkv_par, abort_flag, p.err, kErrB2))) {
        ok = false;
        break;
      }
      dkv_par ^= 1u;
      tc_fence_after();
      const int kvh = hg * kGroupHeads / (p.H / p.Hkv);
      float* wrow =
          p.ws + ((static_cast<long long>(b) * S + (kin ? s : 0)) * p.Hkv + kvh) * (DQK + DV);
#pragma unroll 1
      for (int d0 = 0; d0 < DQK + DV; d0 += 32) {
        uint32_t v[32];
        tmem_ld_x32(tmem + lane_off + L::kColDK + d0, v);
        tmem_ld_wait();
        const float sc = d0 < DQK ? p.scale : 1.f;
        if (kin) {
#pragma unroll
          for (int d = 0; d < 32; d += 4)
            atomicAdd(reinterpret_cast<float4*>(wrow + d0 + d),
                      make_float4(__uint_as_float(v[d]) * sc, __uint_as_float(v[d + 1]) * sc,
                                  __uint_as_float(v[d + 2]) * sc, __uint_as_float(v[d + 3]) * sc));
        }
      }
      tc_fence_before();
      mbar_arrive(&tail->dkv_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

typedef CUresult (*EncodeTiledFnBd)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnBd encode_fn_bd() {
  static EncodeTiledFnBd fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFnBd>(ptr);
  }
  return fn;
}

// K / V [rows, Hkv, cols] bf16 as (column, K/V head, row): boxes of 64 columns x 1 head
// x 128 rows, 128-byte swizzle (the shared-memory tile of a [128 x 64] 2-D box)
bool make_kv_map(CUtensorMap* map, const void* base, long long rows, int Hkv, int cols) {
  EncodeTiledFnBd fn = encode_fn_bd();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                           static_cast<cuuint64_t>(cols) * 2 * static_cast<cuuint64_t>(Hkv)};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kT)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Q / dO [B*S, H, cols] bf16 as (dim, head, row): boxes of 64 dims x 1 head x 64 rows
bool make_head_rows_map(CUtensorMap* map, const void* base, long long rows, int H, int cols) {
  EncodeTiledFnBd fn = encode_fn_bd();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * 2,
                           static_cast<cuuint64_t>(cols) * 2 * static_cast<cuuint64_t>(H)};
  cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(kH)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int DQK, int DV>
int launch_bwd_dense_dims(const AttnParams& p, cudaStream_t stream) {
  using LA = DqLayout<DQK, DV>;
  using LB = DkvLayout<DQK, DV>;
  const int QT = (p.S + kT - 1) / kT;
  const int W4 = QT * 4;
  const long long rows = static_cast<long long>(p.B) * p.S;
  // the bitmap, the tile flags and Delta live in the caller's workspace
  if (p.scratch == nullptr) return DSA_ERR_WORKSPACE;
  const DenseScratch ly = dense_scratch_layout(p.B, p.S, p.H, p.Hkv, DQK, DV, true);
  const size_t any_bytes = static_cast<size_t>(p.B) * QT * QT;
  DenseBwdParams dp;
  dp.a = p;
  dp.bits = reinterpret_cast<uint32_t*>(p.scratch + ly.bits_off);
  dp.any = p.scratch + ly.any_off;
  dp.delta = reinterpret_cast<float*>(p.scratch + ly.delta_off);
  dp.W4 = W4;
  dp.QT = QT;
  CUtensorMap mk, mv, mq, mdo;
  const size_t smem_a = LA::kTailOff + sizeof(DqTail), smem_b = LB::kTailOff + sizeof(DkvTail);
  auto ka = attn_bwd_dense_dq_kernel<DQK, DV>;
  auto kb = attn_bwd_dense_dkv_kernel<DQK, DV>;
  if (cudaMemsetAsync(p.scratch + ly.any_off, 0, any_bytes, stream) != cudaSuccess ||
      !make_kv_map(&mk, p.K, rows, p.Hkv, DQK) || !make_kv_map(&mv, p.V, rows, p.Hkv, DV) ||
      !make_head_rows_map(&mq, p.Q, rows, p.H, DQK) ||
      !make_head_rows_map(&mdo, p.dO, rows, p.H, DV) ||
      cudaFuncSetAttribute(ka, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_a)) != cudaSuccess ||
      cudaFuncSetAttribute(kb, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_b)) != cudaSuccess)
    return DSA_ERR_CUDA;
  launch_dense_mask(p.idx, p.B, p.S, p.k, W4, QT, const_cast<uint32_t*>(dp.bits),
                    const_cast<uint8_t*>(dp.any), p.err, stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long items_a = static_cast<long long>(QT) * p.B * p.H;
  const long long items_b =
      static_cast<long long>(QT) * p.B * ((p.H + kGroupHeads - 1) / kGroupHeads);
  ka<<<static_cast<int>(items_a < sms ? items_a : sms), kThreadsB, smem_a, stream>>>(mk, mv, dp);
  kb<<<static_cast<int>(items_b < sms ? items_b : sms), kThreadsB, smem_b, stream>>>(mk, mv, mq,
                                                                                    mdo, dp);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

bool attn_bwd_dense_supported(int B, int S, int H, int Dqk, int Dv, float scale) {
  const long long items = static_cast<long long>((S + kT - 1) / kT) * B * H;
  return scale > 0.f && S >= 1 && S <= 65536 && H >= 1 && items < (1LL << 31) &&
         ((Dqk == 192 && Dv == 128) || (Dqk == 128 && Dv == 128));
}

// The gathered-key backward costs about one unit per 64-key chunk of a row; a dense
// 128 x 128 tile pair (two 64-key halves in the dq kernel, two 64-query steps in the
// dk/dv kernel) about kDenseBwdTileCost units. Dense when cheaper and the dq kernel's
// items fill the GPU.
bool attn_bwd_dense_preferred(int B, int S, int H, int k) {
  constexpr long long kDenseBwdTileCost = 2;
  const long long QT = (S + kT - 1) / kT;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (QT * B * H < sms) return false;
  const long long dense_units = static_cast<long long>(H) * QT * (QT + 1) / 2;
  const long long N = S < k ? S : k, q = N / 64, rem = N % 64;
  const long long chunks = 64 * q * (q + 1) / 2 + rem * (q + 1) + (S - N) * ((k + 63) / 64);
  (void)B;
  return kDenseBwdTileCost * dense_units < chunks;
}

int launch_attn_bwd_dense(const AttnParams& p, int Dqk, int Dv, cudaStream_t stream) {
  if (Dqk == 192 && Dv == 128) return launch_bwd_dense_dims<192, 128>(p, stream);
  if (Dqk == 128 && Dv == 128) return launch_bwd_dense_dims<128, 128>(p, stream);
  return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
