// Sparse attention forward on the 5th-generation tensor cores, for H <= 128 heads.
//
// ("Support Ring Attention with DeepSeek DSA Sparse Indexer", Forward Flow
// step 5: logits = where(mask, Q K^T * scale, -inf), softmax, P V; the mask is
// the query's selected list intersected with causality.)
//
// All H heads of a query share its selected keys, so the heads are the UMMA M
// dimension (128 TMEM lanes, one head per lane) and the gathered keys are N:
//
//   S_c = Q_t [128 x Dqk] . K_c^T          A = Q from TMEM, B = K_c in smem (K-major)
//   P_c = exp2(S_c * scale*log2e - m)      one softmax thread per head; P -> TMEM (bf16)
//   O  += P_c [128 x NK] . V_c [NK x Dv]   A = P from TMEM, B = V_c in smem (MN-major)
//
// O accumulates in TMEM across the chunks of a row. The running max m used for
// P is refreshed only when a chunk's max exceeds it by more than 2^8 (in exp2
// units); then O and the running sum are rescaled once. Until then P <= 256,
// which bf16 and fp32 hold as well as with a fresh max, and the final O / l is
// unchanged.
//
// Persistent CTA (one per SM), warp-specialised, 384 threads:
//   warps 0-3   softmax / output: Q row -> TMEM, softmax, P -> TMEM, final O and LSE
//   warp  4     TMEM owner and single-thread UMMA issuer
//   warps 5-11  gather: per chunk of NK = 96 selected keys, 16-byte cp.async of the K
//               and V rows into 128B-swizzled tiles (3 stages), four keys per group so
//               that every copy instruction uses all 32 lanes; the copy hardware
//               signals each stage when its rows have landed
// TMEM: [Q: Dqk/2 cols][S/P: 3 buffers x NK cols][O: Dv cols] = 512 columns.
// Query rows are handed out longest first, strided over CTAs.

#include <cstdlib>

#include "dsa_attn_common.cuh"

namespace dsa {
namespace {

constexpr int kNK = 96;              // keys per chunk (UMMA N of S; K of PV)
constexpr int kStages = 3;           // K/V stages == S/P buffers
constexpr int kGatherWarp0 = 5;
constexpr int kGatherWarps = 7;
constexpr int kGatherThreads = 32 * kGatherWarps;
constexpr int kPrefetch = 10;         // index-list entries per gather thread held ahead
constexpr int kThreads = 384;
constexpr int kErrTc = DSA_STAGE_FWD | DSA_DEVERR_TIMEOUT;
constexpr float kRescaleLog2 = 8.f;  // refresh the running max when it grows by > 2^8

template <int DQK, int DV>
struct TcFwdLayout {
  static constexpr int KA = DQK / 64;                 // K atoms (64 dims each)
  static constexpr int VA = DV / 64;                  // V atoms
  static constexpr uint32_t kAtom = kNK * 128;        // one [NK rows x 128 B] atom
  static constexpr uint32_t kStage = (KA + VA) * kAtom;
  static constexpr uint32_t kTailOff = kStages * kStage;
  static constexpr int PIECES = (DQK + DV) / 8;       // 16-byte pieces per key
  static constexpr uint32_t kColQ = 0;
  static constexpr uint32_t kColS = DQK / 2;
  static constexpr uint32_t kColO = kColS + kStages * kNK;
  static_assert(kColO + DV <= 512, "TMEM budget");
};

struct ChunkHeader {
  int row;          // flat query row b*S + t
  int first, last;  // first / last chunk of the row
  int pad;
  uint32_t valid[4];
};

struct TcTail {
  ChunkHeader hdr[kStages];
  int key[kStages][kNK];   // key index per slot of each stage (-1: none)
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[kStages], s_empty[kStages], p_full[kStages];
  uint64_t q_tmem_full, o_free;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int okb[2];
  int red[kGatherWarps];
};

__device__ __forceinline__ void bar_gather() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGatherThreads) : "memory");
}

// Named barrier of the gather threads that also agrees on whether to go on:
// thread 0 samples the abort flag before the barrier and everyone reads that
// one sample after it (two slots, so a fast thread 0 cannot overwrite a verdict
// a slow thread has yet to read).
__device__ __forceinline__ bool bar_gather_ok(int* okb, int& nb, volatile int* abort_flag) {
  if (threadIdx.x == 32 * kGatherWarp0) okb[nb & 1] = (*abort_flag == 0);
  bar_gather();
  const bool ok = reinterpret_cast<volatile int*>(okb)[nb & 1] != 0;
  ++nb;
  return ok;
}

__device__ __forceinline__ long long row_of(int i, int nrows) {
  return static_cast<long long>(nrows) - 1 - i;   // longest rows first
}

__device__ __forceinline__ void drain_wait_tc(uint64_t* bar, uint32_t parity, int* err) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report_error(err, kErrTc);
      return;
    }
  }
}

// key index in slot j of a row, with the causal mask applied; -1 if none
__device__ __forceinline__ int load_key(const AttnParams& p, const int32_t* irow, int j, int kend,
                                        int t) {
  if (j >= kend) return -1;
  int s = __ldg(irow + j);
  if (s < -1 || s >= p.S) {
    report_error(p.err, DSA_STAGE_FWD | DSA_DEVERR_BAD_INDEX);
    s = -1;
  }
  return s > t ? -1 : s;
}

__device__ __forceinline__ void tmem_ld_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int DQK, int DV>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_tc_kernel(const AttnParams p) {
  using L = TcFwdLayout<DQK, DV>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) report_error(p.err, DSA_STAGE_FWD | DSA_DEVERR_MISALIGNED);
    return;
  }
  TcTail* tail = reinterpret_cast<TcTail*>(smem + L::kTailOff);
  volatile int* abort_flag = &tail->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrows = p.B * p.S;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      // per gather thread: one arrive for its header writes, one when its copies land
      mbar_init(&tail->kv_full[i], 2 * kGatherThreads);
      mbar_init(&tail->kv_empty[i], 1);
      mbar_init(&tail->s_full[i], 1);
      mbar_init(&tail->s_empty[i], 1);
      mbar_init(&tail->p_full[i], 128);
    }
    mbar_init(&tail->q_tmem_full, 128);
    mbar_init(&tail->o_free, 128);
    mbar_init(&tail->drain, 1);
    tail->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(&tail->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tail->tmem_base;

  if (warp >= kGatherWarp0) {
    // ================================================================ gather
    // Every gather thread takes part in each step, so the named barriers always
    // see all of them; a timed-out wait sets the abort flag, which all read after
    // the next barrier. Gather thread gt < NK owns key slot gt of every chunk.
    const int gt = threadIdx.x - 32 * kGatherWarp0;
    const int gw = warp - kGatherWarp0;
    constexpr int PK = DQK / 8, PV = DV / 8;     // 16-byte pieces of a K / V row
    constexpr int KI = PK / 8, VI = PV / 8;      // copy instructions per group of 4 keys
    // this lane's (key in group, piece) for each instruction of a group
    int k_kig[KI], k_off[KI], v_kig[VI], v_off[VI];
    uint32_t k_dst[KI], v_dst[VI];
#pragma unroll
    for (int i = 0; i < KI; ++i) {
      const int q = i * 32 + lane, pc = q % PK;
      k_kig[i] = q / PK;
      k_off[i] = pc * 8;
      k_dst[i] = (pc >> 3) * L::kAtom + ((pc & 7) << 4);
    }
#pragma unroll
    for (int i = 0; i < VI; ++i) {
      const int q = i * 32 + lane, pv = q % PV;
      v_kig[i] = q / PV;
      v_off[i] = pv * 8;
      v_dst[i] = (L::KA + (pv >> 3)) * L::kAtom + ((pv & 7) << 4);
    }
    // kend of a row (one past its last slot holding a causal key) needs the whole
    // index list; for k <= kPrefetch * kGatherThreads the next row's list is loaded
    // into registers while the current row is gathered
    const bool prefetch = p.k <= kPrefetch * kGatherThreads;
    int pre[kPrefetch];
    auto load_list = [&](long long row) {
      const int32_t* ir = p.idx + row * p.k;
#pragma unroll
      for (int u = 0; u < kPrefetch; ++u) {
        const int j = gt + u * kGatherThreads;
        pre[u] = j < p.k ? __ldg(ir + j) : -1;
      }
    };
    if (prefetch && static_cast<int>(blockIdx.x) < nrows) load_list(row_of(blockIdx.x, nrows));
    int g = 0, nb = 0;
    for (int i = blockIdx.x; i < nrows; i += gridDim.x) {
      const long long row = row_of(i, nrows);
      const int b = static_cast<int>(row / p.S);
      const int t = static_cast<int>(row - static_cast<long long>(b) * p.S);
      const int32_t* irow = p.idx + row * p.k;
      int last = 0;
      if (prefetch) {
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
          const int s = pre[u];
          if (s >= 0 && s <= t && s < p.S) last = gt + u * kGatherThreads + 1;
        }
        if (i + static_cast<int>(gridDim.x) < nrows) load_list(row_of(i + gridDim.x, nrows));
      } else {
#pragma unroll 10
        for (int j = gt; j < p.k; j += kGatherThreads) {
          const int s = __ldg(irow + j);
          if (s >= 0 && s <= t && s < p.S) last = j + 1;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
      if (lane == 0) tail->red[gw] = last;
      if (!bar_gather_ok(tail->okb, nb, abort_flag)) break;
      int kend = 0;
#pragma unroll
      for (int w2 = 0; w2 < kGatherWarps; ++w2) kend = max(kend, tail->red[w2]);
      const int nch = kend > 0 ? (kend + kNK - 1) / kNK : 1;
      int s_next = gt < kNK ? load_key(p, irow, gt, kend, t) : -1;
      bool stop = false;
      for (int c = 0; c < nch; ++c, ++g) {
        const int st = g % kStages;
        const int s = s_next;
        if (gt < kNK && c + 1 < nch) s_next = load_key(p, irow, (c + 1) * kNK + gt, kend, t);
        mbar_wait(&tail->kv_empty[st], ((g / kStages) & 1) ^ 1u, abort_flag, p.err, kErrTc);
        ChunkHeader& h = tail->hdr[st];
        if (gt < kNK) {
          tail->key[st][gt] = s;
          const uint32_t bal = __ballot_sync(0xffffffffu, s >= 0);
          if (lane == 0) h.valid[gw] = bal;
        }
        if (gt == 0) {
          h.row = static_cast<int>(row);
          h.first = c == 0;
          h.last = c == nch - 1;
        }
        if (!bar_gather_ok(tail->okb, nb, abort_flag)) { stop = true; break; }
        // releases this thread's header writes (the failure-detection test drops the
        // first one of CTA 0, so that the issuer's bounded wait runs out)
        if (!(p.test_drop_arrive && blockIdx.x == 0 && g == 0 && gt == 0))
          mbar_arrive(&tail->kv_full[st]);
        const uint32_t stage = smem_u32(smem + st * L::kStage);
        const long long rowbase = static_cast<long long>(b) * p.S;
        for (int grp = gw; grp < kNK / 4; grp += kGatherWarps) {
          const int4 kq = *reinterpret_cast<const int4*>(&tail->key[st][grp * 4]);
          const int keys[4] = {kq.x, kq.y, kq.z, kq.w};
#pragma unroll
          for (int ii = 0; ii < KI; ++ii) {
            const int kig = k_kig[ii], key = grp * 4 + kig;
            const int ks = kig == 0 ? keys[0] : (kig == 1 ? keys[1] : (kig == 2 ? keys[2] : keys[3]));
            const long long kv = rowbase + (ks >= 0 ? ks : 0);
            const uint32_t dst = stage + key * 128 + (k_dst[ii] ^ ((key & 7) << 4));
            cp_async_16(dst, p.K + kv * DQK + k_off[ii], ks >= 0 ? 16u : 0u);
          }
#pragma unroll
          for (int ii = 0; ii < VI; ++ii) {
            const int kig = v_kig[ii], key = grp * 4 + kig;
            const int ks = kig == 0 ? keys[0] : (kig == 1 ? keys[1] : (kig == 2 ? keys[2] : keys[3]));
            const long long kv = rowbase + (ks >= 0 ? ks : 0);
            const uint32_t dst = stage + key * 128 + (v_dst[ii] ^ ((key & 7) << 4));
            cp_async_16(dst, p.V + kv * DV + v_off[ii], ks >= 0 ? 16u : 0u);
          }
        }
        // second arrival, made by the copy hardware once this thread's copies have landed
        cp_async_mbar_arrive(&tail->kv_full[st]);
      }
      if (stop) break;
    }
    cp_async_wait<0>();
  } else if (warp == 4) {
    // ================================================================ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16_mn(128, kNK, false);
      constexpr uint32_t idesc_pv = umma_idesc_bf16_mn(128, DV, true);
      int g = 0;
      uint32_t qt_par = 0, of_par = 1;
      int pend = -1, pend_first = 0;   // chunk whose PV is still to be issued
      bool ok = true;
      for (int i = blockIdx.x; ok && i < nrows; i += gridDim.x) {
        bool last = false;
        while (ok && !last) {
          const int sb = g % kStages;
          const uint32_t use_par = (g / kStages) & 1;
          if (!mbar_wait(&tail->kv_full[sb], use_par, abort_flag, p.err, kErrTc)) { ok = false; break; }
          const ChunkHeader& h = tail->hdr[sb];
          last = h.last != 0;
          const int first = h.first;
          if (first) {
            if (!mbar_wait(&tail->q_tmem_full, qt_par, abort_flag, p.err, kErrTc)) { ok = false; break; }
            qt_par ^= 1u;
          }
          if (!mbar_wait(&tail->s_empty[sb], use_par ^ 1u, abort_flag, p.err, kErrTc)) { ok = false; break; }
          // K/V rows were written by cp.async (generic proxy); the tensor cores read
          // them through the async proxy
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t kbase = smem_u32(smem + sb * L::kStage);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint64_t bdesc =
                umma_sdesc(kbase + (kk >> 2) * L::kAtom + (kk & 3) * 32, 1024, kLayoutSw128);
            umma_bf16_ts(tmem + L::kColS + sb * kNK, tmem + L::kColQ + kk * 8, bdesc, idesc_s,
                         kk > 0 ? 1u : 0u);
          }
          umma_commit(&tail->s_full[sb]);
          if (pend >= 0) {
            // PV of the previous chunk, once its P is in TMEM
            const int pb = pend % kStages;
            if (!mbar_wait(&tail->p_full[pb], (pend / kStages) & 1, abort_flag, p.err, kErrTc)) { ok = false; break; }
            if (pend_first) {   // the previous row's O has been read out
              if (!mbar_wait(&tail->o_free, of_par, abort_flag, p.err, kErrTc)) { ok = false; break; }
              of_par ^= 1u;
            }
            tc_fence_after();
            const uint32_t vbase = smem_u32(smem + pb * L::kStage + L::KA * L::kAtom);
#pragma unroll
            for (int ks = 0; ks < kNK / 16; ++ks) {
              const uint64_t bdesc =
                  umma_sdesc_lbo(vbase + ks * 2048, L::kAtom, 1024, kLayoutSw128);
              umma_bf16_ts(tmem + L::kColO, tmem + L::kColS + pb * kNK + ks * 8, bdesc, idesc_pv,
                           (pend_first && ks == 0) ? 0u : 1u);
            }
            umma_commit(&tail->kv_empty[pb]);
            umma_commit(&tail->s_empty[pb]);
          }
          if (last) {
            // the row's last chunk: its PV right away, so that the row's O is
            // complete before the next row's first chunk arrives
            const int pb = sb;
            if (!mbar_wait(&tail->p_full[pb], use_par, abort_flag, p.err, kErrTc)) { ok = false; break; }
            if (first) {
              if (!mbar_wait(&tail->o_free, of_par, abort_flag, p.err, kErrTc)) { ok = false; break; }
              of_par ^= 1u;
            }
            tc_fence_after();
            const uint32_t vbase = smem_u32(smem + pb * L::kStage + L::KA * L::kAtom);
#pragma unroll
            for (int ks = 0; ks < kNK / 16; ++ks) {
              const uint64_t bdesc =
                  umma_sdesc_lbo(vbase + ks * 2048, L::kAtom, 1024, kLayoutSw128);
              umma_bf16_ts(tmem + L::kColO, tmem + L::kColS + pb * kNK + ks * 8, bdesc, idesc_pv,
                           (first && ks == 0) ? 0u : 1u);
            }
            umma_commit(&tail->kv_empty[pb]);
            umma_commit(&tail->s_empty[pb]);
            pend = -1;
          } else {
            pend = g;
            pend_first = first;
          }
          ++g;
        }
      }
      if (ok && pend >= 0) {
        const int pb = pend % kStages;
        bool go = mbar_wait(&tail->p_full[pb], (pend / kStages) & 1, abort_flag, p.err, kErrTc);
        if (go && pend_first) {
          go = mbar_wait(&tail->o_free, of_par, abort_flag, p.err, kErrTc);
          of_par ^= 1u;
        }
        if (go) {
          tc_fence_after();
          const uint32_t vbase = smem_u32(smem + pb * L::kStage + L::KA * L::kAtom);
#pragma unroll
          for (int ks = 0; ks < kNK / 16; ++ks) {
            const uint64_t bdesc = umma_sdesc_lbo(vbase + ks * 2048, L::kAtom, 1024, kLayoutSw128);
            umma_bf16_ts(tmem + L::kColO, tmem + L::kColS + pb * kNK + ks * 8, bdesc, idesc_pv,
                         (pend_first && ks == 0) ? 0u : 1u);
          }
          umma_commit(&tail->kv_empty[pb]);
          umma_commit(&tail->s_empty[pb]);
        }
      }
      umma_commit(&tail->drain);
      drain_wait_tc(&tail->drain, 0, p.err);
    }
  } else {
    // ================================================================ softmax / output
    const int quarter = warp;                              // warps 0-3: TMEM lane quarters
    const int hrow = quarter * 32 + lane;                  // head of this thread
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float c2 = p.scale_log2;
    const int H = p.H;
    const long long qrows = static_cast<long long>(nrows) * H;
    int g = 0;
    bool ok = true;

    // Q row of this thread's head -> its TMEM lane as packed bf16 pairs. Lanes
    // >= H read the following rows of Q (zeros past the end): computed, never stored.
    auto load_q = [&](long long row) {
      const long long qrow = row * H + hrow;
      const bool in = qrow < qrows;
      const uint4* src = reinterpret_cast<const uint4*>(p.Q + (in ? qrow : 0) * DQK);
#pragma unroll
      for (int a = 0; a < DQK / 64; ++a) {
        uint32_t lo[16], hi[16];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint4 x = in ? __ldg(src + a * 8 + cc) : make_uint4(0, 0, 0, 0);
          const uint4 y = in ? __ldg(src + a * 8 + 4 + cc) : make_uint4(0, 0, 0, 0);
          lo[cc * 4 + 0] = x.x; lo[cc * 4 + 1] = x.y; lo[cc * 4 + 2] = x.z; lo[cc * 4 + 3] = x.w;
          hi[cc * 4 + 0] = y.x; hi[cc * 4 + 1] = y.y; hi[cc * 4 + 2] = y.z; hi[cc * 4 + 3] = y.w;
        }
        tmem_st_x16(tmem + lane_off + L::kColQ + a * 32, lo);
        tmem_st_x16(tmem + lane_off + L::kColQ + a * 32 + 16, hi);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&tail->q_tmem_full);
    };

    if (static_cast<int>(blockIdx.x) < nrows) load_q(row_of(blockIdx.x, nrows));
    for (int i = blockIdx.x; ok && i < nrows; i += gridDim.x) {
      float m = -INFINITY, l = 0.f;   // running max (raw logits) and sum
      bool last = false;
      int row = 0;
      while (!last) {
        const int sb = g % kStages;
        const uint32_t use_par = (g / kStages) & 1;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tail->s_full[sb], use_par, abort_flag, p.err, kErrTc))) {
          ok = false;
          break;
        }
        // acquire the gather threads' header writes (this phase cannot advance
        // before this chunk's P has been consumed)
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tail->kv_full[sb], use_par, abort_flag, p.err, kErrTc))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const ChunkHeader& h = tail->hdr[sb];
        last = h.last != 0;
        const bool first = h.first != 0;
        row = h.row;
        const uint32_t vm0 = h.valid[0], vm1 = h.valid[1], vm2 = h.valid[2];
        const bool all_valid = (vm0 & vm1 & vm2) == 0xffffffffu;
        const uint32_t sbase = tmem + lane_off + L::kColS + sb * kNK;
        // the chunk's maximum over its valid keys, 32 columns at a time; S is read from TMEM
        // again for the exponentials, so that no 96 logits are held in registers (TMEM loads
        // are cheap, and the kernel then fits its registers without spilling)
        float mx = -INFINITY;
#pragma unroll 1
        for (int part = 0; part < 3; ++part) {
          uint32_t sv[32];
          tmem_ld_x32(sbase + part * 32, sv);
          tmem_ld_wait();
          const uint32_t vm = part == 0 ? vm0 : (part == 1 ? vm1 : vm2);
          if (all_valid) {
#pragma unroll
            for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(sv[j]));
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if ((vm >> j) & 1u) mx = fmaxf(mx, __uint_as_float(sv[j]));
          }
        }
        if (first) {
          m = mx;
        } else if (__any_sync(0xffffffffu,
                              mx > m && (m == -INFINITY || (mx - m) * c2 > kRescaleLog2))) {
          // refresh the running max of every head of the warp (a no-op where it has
          // not grown): rescale O (every earlier PV product is done) and l
          const int pg = g - 1;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&tail->s_empty[pg % kStages], (pg / kStages) & 1, abort_flag,
                                    p.err, kErrTc))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float mnew = fmaxf(m, mx);
          const float f = m == -INFINITY ? 0.f : exp2f((m - mnew) * c2);
#pragma unroll
          for (int d0 = 0; d0 < DV; d0 += 16) {
            uint32_t ov[16];
            tmem_ld_x16(tmem + lane_off + L::kColO + d0, ov);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * f);
            tmem_st_x16(tmem + lane_off + L::kColO + d0, ov);
          }
          tmem_st_wait();
          l *= f;
          m = mnew;
        }
        // P = exp2(S*c2 - m*c2) over valid keys -> bf16 pairs in the buffer's first NK/2 cols
        const float base = m == -INFINITY ? 0.f : m * c2;
        float ls = 0.f;
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          uint32_t sv[32];
          tmem_ld_x32(sbase + part * 32, sv);
          tmem_ld_wait();
          const uint32_t vm = part == 0 ? vm0 : (part == 1 ? vm1 : vm2);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float e0 = ex2(fmaf(__uint_as_float(sv[j]), c2, -base));
            float e1 = ex2(fmaf(__uint_as_float(sv[j + 1]), c2, -base));
            if (!all_valid) {
              e0 = ((vm >> j) & 1u) ? e0 : 0.f;
              e1 = ((vm >> (j + 1)) & 1u) ? e1 : 0.f;
            }
            ls += e0 + e1;
            pk[j >> 1] = pack_bf16(e0, e1);
          }
          tmem_st_x16(sbase + part * 16, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&tail->p_full[sb]);
        l += ls;
        if (last && i + static_cast<int>(gridDim.x) < nrows) {
          // every S of this row is done: the next row's Q may replace it in TMEM
          load_q(row_of(i + gridDim.x, nrows));
        }
        ++g;
      }
      if (!ok) break;
      // final O: wait for this row's last PV, normalise, store; then release O
      const int pg = g - 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&tail->s_empty[pg % kStages], (pg / kStages) & 1,
                                              abort_flag, p.err, kErrTc))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* orow = reinterpret_cast<uint4*>(p.O + (static_cast<long long>(row) * H + hrow) * DV);
#pragma unroll
      for (int d0 = 0; d0 < DV; d0 += 32) {
        uint32_t ov[32];
        tmem_ld_x32(tmem + lane_off + L::kColO + d0, ov);
        tmem_ld_wait();
        if (hrow < H) {
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
      if (hrow < H)
        p.lse[static_cast<long long>(row) * H + hrow] =
            l > 0.f ? (m * c2 + log2f(l)) * 0.69314718055994530942f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, 512);
}

template <int DQK, int DV>
int launch_tc(const AttnParams& p, cudaStream_t stream) {
  using L = TcFwdLayout<DQK, DV>;
  const size_t smem = L::kTailOff + sizeof(TcTail);
  auto kern = attn_fwd_tc_kernel<DQK, DV>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long rows = static_cast<long long>(p.B) * p.S;
  const int grid = static_cast<int>(rows < sms ? rows : sms);
  // Failure-detection test: with DSA_TEST_DROP_ARRIVE set in the environment
  // when the library first launches this kernel, one producer arrive is skipped
  // and the call ends through the bounded-wait timeout path.
  static const int drop = std::getenv("DSA_TEST_DROP_ARRIVE") != nullptr ? 1 : 0;
  AttnParams q = p;
  q.test_drop_arrive = drop;
  kern<<<grid, kThreads, smem, stream>>>(q);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

// Any H <= 128: the heads fill TMEM lanes 0..H-1 and the lanes above compute on
// the following query rows' Q (or zeros) and store nothing. With few heads most of
// the M = 128 tile is idle, but the kernel is bound by its per-chunk pipeline and
// the K/V gather rather than by the tensor cores.
bool attn_fwd_tc_supported(int H, int Dqk, int Dv, float scale) {
  return H >= 1 && H <= 128 && scale > 0.f &&
         ((Dqk == 192 && Dv == 128) || (Dqk == 128 && Dv == 128));
}

int launch_attn_fwd_tc(const AttnParams& p, int Dqk, int Dv, cudaStream_t stream) {
  if (Dqk == 192 && Dv == 128) return launch_tc<192, 128>(p, stream);
  if (Dqk == 128 && Dv == 128) return launch_tc<128, 128>(p, stream);
  return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
