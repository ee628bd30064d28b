// Sparse attention backward on the 5th-generation tensor cores, for H <= 128 heads.
//
// ("Support Ring Attention with DeepSeek DSA Sparse Indexer", Backward Flow
// step 6: dQ = dP K, dK = dP^T Q, dV = P^T dO over the same mask, "dP" read as
// the gradient of the logits.)
//
// Per query row t (all heads; the row's selected keys in chunks of NK = 64):
//
//   S   = Q . K_c^T            M = heads, N = keys   A = Q   (smem, K-major)   B = K_c (K-major)
//   dP  = dO . V_c^T           M = heads, N = keys   A = dO  (smem, K-major)   B = V_c (K-major)
//   P   = exp2(S*scale*log2e - lse*log2e), dS = P (dP - Delta)      softmax warps -> bf16 tiles
//   dQ += dS . K_c             M = heads, N = Dqk    A = dS  (smem, K-major)   B = K_c (MN-major)
//   dK_c^T = Q^T . dS          M = dims,  N = keys   A = Q   (smem, MN-major)  B = dS  (MN-major)
//   dV_c^T = dO^T . P          M = dims,  N = keys   A = dO  (smem, MN-major)  B = P   (MN-major)
//
// The same shared tiles serve as K-major and MN-major operands. dK/dV are
// produced transposed (a TMEM lane per dimension), so the fp32 reductions
// that add them into the [B*S, Dqk+Dv] accumulator are row-contiguous: a warp
// covers 32 consecutive floats of one key row per instruction. dQ stays in
// TMEM for the whole row. Delta = sum_c dO O is formed at the start of each row.
//
// Persistent CTA (one per SM), 512 threads:
//   warps 0-3   softmax: Delta, P and dS tiles, final dQ (one head per thread)
//   warps 4-11  drain: dK^T / dV^T from TMEM -> fp32 reductions (one dim per thread;
//               two warps per TMEM lane quarter, one per half of the chunk's keys)
//   warp  12    TMEM owner; issues S and dP, and loads each row's Q / dO tiles (TMA)
//               once the previous row's gradient MMAs have released them
//   warp  13    issues dQ, dK^T and dV^T (in that order: dV^T, the one product that
//               reads P, comes last, and dS is double-buffered, so the softmax warps
//               write the next chunk's dS while this chunk's products still run)
//   warps 14-15 gather: K/V rows of each chunk (cp.async, 2 stages; a stage is
//               released as soon as the chunk's dQ product has read it)
// TMEM: dQ [0,192) S [192,256) dP [256,320) dK^T lo [320,384) hi [384,448) dV^T [448,512).

#include "dsa_attn_common.cuh"

namespace dsa {
namespace {

constexpr int NK = 64;               // keys per chunk
constexpr int kStages = 2;           // K/V gather stages
constexpr int kKeyRing = 4;          // key lists of chunks in flight
constexpr int kDrainWarps = 8;
constexpr int kMmaWarp = 12;        // TMEM owner, Q / dO loads, S and dP MMAs
constexpr int kGradWarp = 13;        // dQ, dK^T, dV^T MMAs
constexpr int kGatherWarp0 = 14;
constexpr int kGatherWarps = 2;
constexpr int kGatherThreads = 32 * kGatherWarps;
static_assert(kGatherThreads >= 64, "a gather thread per key slot");
constexpr int kPrefetch = 32;        // index-list entries per gather thread held ahead
constexpr int kThreads = 512;
constexpr int kErrB = DSA_STAGE_BWD | DSA_DEVERR_TIMEOUT;

// Dqk = 192, Dv = 128
constexpr int DQK = 192, DV = 128;
constexpr uint32_t kQAtom = 128 * 128;           // [128 head rows x 64 dims]
constexpr uint32_t kQOff = 0;                    // 3 atoms
constexpr uint32_t kDOOff = 3 * kQAtom;          // 2 atoms, right after Q
constexpr uint32_t kKVAtom = NK * 128;           // [64 key rows x 64 dims]
constexpr uint32_t kKVStage = 5 * kKVAtom;       // K: 3 atoms, V: 2 atoms
constexpr uint32_t kKVOff = kDOOff + 2 * kQAtom;
constexpr uint32_t kPOff = kKVOff + kStages * kKVStage;   // [128 heads x 64 keys]
constexpr uint32_t kDSOff = kPOff + kQAtom;                  // 2 buffers (chunk parity)
constexpr uint32_t kDrainOff = kDSOff + 2 * kQAtom;          // per drain warp: [16 keys x 32]
constexpr int kDrainPitch = 32;   // floats; a quarter-warp reads one 128-byte row: no conflicts
constexpr uint32_t kDrainTile = 16 * kDrainPitch * 4;
constexpr uint32_t kTailOff = kDrainOff + kDrainWarps * kDrainTile;
static_assert(kTailOff + 2048 <= 232448, "shared memory: tiles + tail within 227 KB");
constexpr uint32_t kColDQ = 0, kColS = 192, kColDP = 256, kColDKlo = 320, kColDKhi = 384,
                   kColDV = 448;

struct BwdTail {
  int key[kKeyRing][NK];       // key index per slot (-1: none)
  int row[kKeyRing];
  int flags[kKeyRing];         // bit 0: first chunk of row, bit 1: last
  uint32_t valid[kKeyRing][2];
  uint64_t keys_full[kKeyRing];   // the key list / flags of a ring slot are written
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t qdo_full, qdo_free;
  uint64_t sdp_full, sdp_free;
  uint64_t ds_full[2], ds_free[2];   // dS tiles, double-buffered by chunk parity
  uint64_t p_full, p_free;           // the P tile
  uint64_t dkv_full[3], dkv_free[3];   // per region: dV^T, dK^T lo, dK^T hi
  uint64_t dq_full, dq_free;
  uint64_t drain, drain_g;
  uint32_t tmem_base;
  int abort_flag;
  int okb[2];
  int red[kGatherWarps];
};

__device__ __forceinline__ void bar_gather() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGatherThreads) : "memory");
}

__device__ __forceinline__ bool bar_gather_ok(int* okb, int& nb, volatile int* abort_flag) {
  if (threadIdx.x == 32 * kGatherWarp0) okb[nb & 1] = (*abort_flag == 0);
  bar_gather();
  const bool ok = reinterpret_cast<volatile int*>(okb)[nb & 1] != 0;
  ++nb;
  return ok;
}

__device__ __forceinline__ long long brow_of(int i, int nrows) {
  return static_cast<long long>(nrows) - 1 - i;
}

__device__ __forceinline__ void drain_wait_b(uint64_t* bar, uint32_t parity, int* err) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report_error(err, kErrB);
      return;
    }
  }
}

__device__ __forceinline__ int load_key_b(const AttnParams& p, const int32_t* irow, int j,
                                          int kend, int t) {
  if (j >= kend) return -1;
  int s = __ldg(irow + j);
  if (s < -1 || s >= p.S) {
    report_error(p.err, DSA_STAGE_BWD | DSA_DEVERR_BAD_INDEX);
    s = -1;
  }
  return s > t ? -1 : s;
}

__device__ __forceinline__ void tmem_ld_x16_b(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ float ex2b(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t acc) {
  umma_bf16(d, a, b, idesc, acc);
}

// instruction descriptor with both major bits
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn ? (1u << 15) : 0u) |
         (b_mn ? (1u << 16) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_do, const AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) report_error(p.err, DSA_STAGE_BWD | DSA_DEVERR_MISALIGNED);
    return;
  }
  BwdTail* tail = reinterpret_cast<BwdTail*>(smem + kTailOff);
  volatile int* abort_flag = &tail->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrows = p.B * p.S;
  const int H = p.H;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&tail->kv_full[i], 2 * kGatherThreads);
      mbar_init(&tail->kv_empty[i], 1);
    }
    for (int i = 0; i < kKeyRing; ++i) mbar_init(&tail->keys_full[i], kGatherThreads);
    mbar_init(&tail->qdo_full, 1);
    mbar_init(&tail->qdo_free, 1);
    mbar_init(&tail->sdp_full, 1);
    mbar_init(&tail->sdp_free, 128);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tail->ds_full[i], 128);
      mbar_init(&tail->ds_free[i], 1);
    }
    mbar_init(&tail->p_full, 128);
    mbar_init(&tail->p_free, 1);
    for (int r = 0; r < 3; ++r) {
      mbar_init(&tail->dkv_full[r], 1);
      mbar_init(&tail->dkv_free[r], 32 * kDrainWarps);
    }
    mbar_init(&tail->dq_full, 1);
    mbar_init(&tail->dq_free, 128);
    mbar_init(&tail->drain, 1);
    mbar_init(&tail->drain_g, 1);
    tail->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tail->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tail->tmem_base;

  if (warp >= kGatherWarp0) {
    // ================================================================ gather
    const int gt = threadIdx.x - 32 * kGatherWarp0;   // 0..95; gt < NK owns key slot gt
    const int gw = warp - kGatherWarp0;
    // a warp copies 4 keys at a time: 8 lanes per key, one 16-byte piece of each
    // 64-dim atom row per lane (K: 3 atoms, V: 2), 4 x 128 contiguous bytes per instruction
    const int sub = lane >> 3, pc = lane & 7;
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
    if (prefetch && static_cast<int>(blockIdx.x) < nrows) load_list(brow_of(blockIdx.x, nrows));
    int g = 0, nb = 0;
    for (int i = blockIdx.x; i < nrows; i += gridDim.x) {
      const long long row = brow_of(i, nrows);
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
        if (i + static_cast<int>(gridDim.x) < nrows) load_list(brow_of(i + gridDim.x, nrows));
      } else {
#pragma unroll 8
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
      const int nch = kend > 0 ? (kend + NK - 1) / NK : 1;
      int s_next = gt < NK ? load_key_b(p, irow, gt, kend, t) : -1;
      bool stop = false;
      for (int c = 0; c < nch; ++c, ++g) {
        const int st = g % kStages, kr = g % kKeyRing;
        const int s = s_next;
        if (gt < NK && c + 1 < nch) s_next = load_key_b(p, irow, (c + 1) * NK + gt, kend, t);
        mbar_wait(&tail->kv_empty[st], ((g / kStages) & 1) ^ 1u, abort_flag, p.err, kErrB);
        if (gt < NK) {
          tail->key[kr][gt] = s;
          const uint32_t bal = __ballot_sync(0xffffffffu, s >= 0);
          if (lane == 0) tail->valid[kr][gw] = bal;
        }
        if (gt == 0) {
          tail->row[kr] = static_cast<int>(row);
          tail->flags[kr] = (c == 0 ? 1 : 0) | (c == nch - 1 ? 2 : 0);
        }
        if (!bar_gather_ok(tail->okb, nb, abort_flag)) { stop = true; break; }
        mbar_arrive(&tail->keys_full[kr]);   // releases this thread's list writes
        mbar_arrive(&tail->kv_full[st]);
        const uint32_t stage = smem_u32(smem + kKVOff + st * kKVStage);
        const long long rowbase = static_cast<long long>(b) * p.S;
        for (int grp = gw; grp < NK / 4; grp += kGatherWarps) {
          const int slot = grp * 4 + sub;
          const int ks = tail->key[kr][slot];
          const long long kv = rowbase + (ks >= 0 ? ks : 0);
          const uint32_t n = ks >= 0 ? 16u : 0u;   // 0: zero-fill an empty slot
          const auto* ksrc = p.K + kv * DQK + pc * 8;
          const auto* vsrc = p.V + kv * DV + pc * 8;
          const uint32_t dst = stage + slot * 128 + ((pc ^ (slot & 7)) << 4);
#pragma unroll
          for (int a = 0; a < 3; ++a) cp_async_16(dst + a * kKVAtom, ksrc + a * 64, n);
#pragma unroll
          for (int a = 0; a < 2; ++a) cp_async_16(dst + (3 + a) * kKVAtom, vsrc + a * 64, n);
        }
        cp_async_mbar_arrive(&tail->kv_full[st]);
      }
      if (stop) break;
    }
    cp_async_wait<0>();
  } else if (warp == kMmaWarp || warp == kGradWarp) {
    // ================================================================ UMMA issuers
    // Two issuing threads keep the tensor pipe fed while either waits: warp 12 issues
    // S / dP (and loads each row's Q / dO), warp 13 the gradients. A commit tracks the
    // committing thread's own MMAs; the gradient MMAs of a chunk start only after its
    // dS exists, so the S / dP MMAs that read the same K / V stage are complete then.
    if (lane == 0) {
      constexpr uint32_t id_sdp = idesc_bf16(128, NK, false, false);
      constexpr uint32_t id_dq = idesc_bf16(128, DQK, false, true);
      constexpr uint32_t id_dkv = idesc_bf16(128, NK, true, true);
      const uint32_t q_s = smem_u32(smem + kQOff), do_s = smem_u32(smem + kDOOff);
      const uint32_t p_s = smem_u32(smem + kPOff), ds_s = smem_u32(smem + kDSOff);
      const uint32_t kv0 = smem_u32(smem + kKVOff);
      // base descriptors, built once; every MMA below advances one by a constant
      const uint64_t q_k = umma_sdesc(q_s, 1024, kLayoutSw128);      // K-major operands
      const uint64_t do_k = umma_sdesc(do_s, 1024, kLayoutSw128);
      const uint64_t ds_k = umma_sdesc(ds_s, 1024, kLayoutSw128);
      const uint64_t kv_k = umma_sdesc(kv0, 1024, kLayoutSw128);
      const uint64_t kv_mn = umma_sdesc_lbo(kv0, kKVAtom, 1024, kLayoutSw128);   // MN-major
      const uint64_t q_mn = umma_sdesc_lbo(q_s, kQAtom, 1024, kLayoutSw128);
      const uint64_t do_mn = umma_sdesc_lbo(do_s, kQAtom, 1024, kLayoutSw128);
      const uint64_t p_mn = umma_sdesc_lbo(p_s, kQAtom, 1024, kLayoutSw128);
      const uint64_t ds_mn = umma_sdesc_lbo(ds_s, kQAtom, 1024, kLayoutSw128);
      const uint64_t q_hi_mn = umma_desc_adv(q_mn, 2 * kQAtom);
      int g = 0, nrow = 0;
      bool ok = true;
      // dQ, dK^T, dV^T of chunk pg (its P / dS tiles are ready); prow = its row ordinal
      // The next chunk's dS goes to the other buffer, so its dQ / dK^T MMAs can follow
      // this chunk's at once; only dV^T (the one product that reads P) waits for the
      // single P tile.
      auto issue_grads = [&](int pg, int flags, int prow) -> bool {
        const int st = pg % kStages, db = pg & 1;
        if (!mbar_wait(&tail->ds_full[db], (pg >> 1) & 1, abort_flag, p.err, kErrB)) return false;
        if ((flags & 1) &&   // first chunk of a row: the previous row's dQ was read out
            !mbar_wait(&tail->dq_free, (prow & 1) ^ 1u, abort_flag, p.err, kErrB))
          return false;
        tc_fence_after();
        const uint64_t kst_mn = umma_desc_adv(kv_mn, st * kKVStage);
        const uint64_t dsb_k = umma_desc_adv(ds_k, db * kQAtom);
        const uint64_t dsb_mn = umma_desc_adv(ds_mn, db * kQAtom);
#pragma unroll
        for (int kk = 0; kk < NK / 16; ++kk) {
          umma_ss(tmem + kColDQ, umma_desc_adv(dsb_k, kk * 32), umma_desc_adv(kst_mn, kk * 2048),
                  id_dq, ((flags & 1) && kk == 0) ? 0u : 1u);
        }
        if (flags & 2) umma_commit(&tail->dq_full);
        umma_commit(&tail->kv_empty[st]);   // K / V of this stage are no longer read
        // dK^T lo, dK^T hi, dV^T, each once the drain warps have emptied that region of
        // the previous chunk (so draining and MMAs overlap by region); unrolled, so that
        // each MMA is a constant advance of a base descriptor
#pragma unroll
        for (int ri = 0; ri < 3; ++ri) {
          const int reg = ri == 2 ? 0 : ri + 1;
          if (reg == 0) {
            umma_commit(&tail->ds_free[db]);
            if (!mbar_wait(&tail->p_full, pg & 1, abort_flag, p.err, kErrB)) return false;
          }
          if (!mbar_wait(&tail->dkv_free[reg], (pg & 1) ^ 1u, abort_flag, p.err, kErrB)) return false;
          tc_fence_after();
          const uint32_t dcol = reg == 0 ? kColDV : (reg == 1 ? kColDKlo : kColDKhi);
          const uint64_t ad = reg == 0 ? do_mn : (reg == 1 ? q_mn : q_hi_mn);
          const uint64_t bd = reg == 0 ? p_mn : dsb_mn;
#pragma unroll
          for (int kk = 0; kk < 128 / 16; ++kk)
            umma_ss(tmem + dcol, umma_desc_adv(ad, kk * 2048), umma_desc_adv(bd, kk * 2048), id_dkv,
                    kk > 0 ? 1u : 0u);
          umma_commit(&tail->dkv_full[reg]);
        }
        umma_commit(&tail->p_free);
        if (flags & 2) umma_commit(&tail->qdo_free);
        return true;
      };
      if (warp == kGradWarp) {
        // chunks in order, their flags from the key ring
        for (int i = blockIdx.x; ok && i < nrows; i += gridDim.x, ++nrow) {
          bool last = false;
          while (ok && !last) {
            const int kr = g % kKeyRing;
            if (!mbar_wait(&tail->keys_full[kr], (g / kKeyRing) & 1, abort_flag, p.err, kErrB)) {
              ok = false;
              break;
            }
            const int flags = tail->flags[kr];
            last = (flags & 2) != 0;
            if (!issue_grads(g, flags, nrow)) { ok = false; break; }
            ++g;
          }
        }
        umma_commit(&tail->drain_g);
        drain_wait_b(&tail->drain_g, 0, p.err);
      } else {
        for (int i = blockIdx.x; ok && i < nrows; i += gridDim.x, ++nrow) {
          bool last = false;
          while (ok && !last) {
            const int st = g % kStages, kr = g % kKeyRing;
            if (!mbar_wait(&tail->kv_full[st], (g / kStages) & 1, abort_flag, p.err, kErrB)) { ok = false; break; }
            const int flags = tail->flags[kr];
            last = (flags & 2) != 0;
            if (flags & 1) {
              // a new row: once the previous row's gradient MMAs are done its Q / dO
              // tiles can be replaced by this row's (TMA)
              if (nrow > 0 &&
                  !mbar_wait(&tail->qdo_free, (nrow - 1) & 1, abort_flag, p.err, kErrB)) { ok = false; break; }
              mbar_arrive_expect_tx(&tail->qdo_full, 5 * kQAtom);
              const int qrow = tail->row[kr] * H;
#pragma unroll
              for (int a = 0; a < 3; ++a)
                tma_load_2d(smem + kQOff + a * kQAtom, &tm_q, &tail->qdo_full, a * 64, qrow);
#pragma unroll
              for (int a = 0; a < 2; ++a)
                tma_load_2d(smem + kDOOff + a * kQAtom, &tm_do, &tail->qdo_full, a * 64, qrow);
              if (!mbar_wait(&tail->qdo_full, nrow & 1, abort_flag, p.err, kErrB)) {
                drain_wait_b(&tail->qdo_full, nrow & 1, p.err);   // let the copy land before exit
                ok = false;
                break;
              }
            }
            // S / dP of this chunk need the softmax warps to have read the previous ones
            if (g > 0 && !mbar_wait(&tail->sdp_free, (g - 1) & 1, abort_flag, p.err, kErrB)) { ok = false; break; }
            fence_proxy_async_smem();
            tc_fence_after();
            const uint64_t kst_k = umma_desc_adv(kv_k, st * kKVStage);
#pragma unroll
            for (int kk = 0; kk < DQK / 16; ++kk)
              umma_ss(tmem + kColS, umma_desc_adv(q_k, (kk >> 2) * kQAtom + (kk & 3) * 32),
                      umma_desc_adv(kst_k, (kk >> 2) * kKVAtom + (kk & 3) * 32), id_sdp,
                      kk > 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < DV / 16; ++kk)
              umma_ss(tmem + kColDP, umma_desc_adv(do_k, (kk >> 2) * kQAtom + (kk & 3) * 32),
                      umma_desc_adv(kst_k, (3 + (kk >> 2)) * kKVAtom + (kk & 3) * 32), id_sdp,
                      kk > 0 ? 1u : 0u);
            umma_commit(&tail->sdp_full);
            ++g;
          }
        }
        umma_commit(&tail->drain);
        drain_wait_b(&tail->drain, 0, p.err);
      }
    }
  } else if (warp < 4) {
    // ================================================================ softmax
    const int hrow = warp * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const float c2 = p.scale_log2;
    uint8_t* prow = smem + kPOff + hrow * 128;
    uint8_t* dsrow0 = smem + kDSOff + hrow * 128;
    const uint32_t sw = static_cast<uint32_t>(hrow & 7);
    int g = 0, nrow = 0;
    bool ok = true;
    for (int i = blockIdx.x; ok && i < nrows; i += gridDim.x, ++nrow) {
      const long long row = brow_of(i, nrows);
      const bool hv = hrow < H;
      // Delta = sum_c dO[c] O[c] and lse of this head (fp32)
      float delta = 0.f, lse2 = 0.f;
      if (hv) {
        const uint4* o4 = reinterpret_cast<const uint4*>(p.O_in + (row * H + hrow) * DV);
        const uint4* d4 = reinterpret_cast<const uint4*>(p.dO + (row * H + hrow) * DV);
#pragma unroll 4
        for (int j = 0; j < DV / 8; ++j) {
          const uint4 a = __ldg(o4 + j), d = __ldg(d4 + j);
          const uint32_t av[4] = {a.x, a.y, a.z, a.w}, dv[4] = {d.x, d.y, d.z, d.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            delta = fmaf(__uint_as_float(av[e] << 16), __uint_as_float(dv[e] << 16), delta);
            delta = fmaf(__uint_as_float(av[e] & 0xffff0000u), __uint_as_float(dv[e] & 0xffff0000u),
                         delta);
          }
        }
        lse2 = p.lse_in[row * H + hrow] * 1.4426950408889634f;
      }
      bool last = false;
      while (!last) {
        const int kr = g % kKeyRing;
        if (!__all_sync(0xffffffffu, mbar_wait(&tail->sdp_full, g & 1, abort_flag, p.err, kErrB))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // acquire the gather threads' list writes (the slot is not rewritten before
        // this chunk's P / dS have been consumed)
        if (!__all_sync(0xffffffffu, mbar_wait(&tail->keys_full[kr], (g / kKeyRing) & 1,
                                                abort_flag, p.err, kErrB))) {
          ok = false;
          break;
        }
        last = (tail->flags[kr] & 2) != 0;
        const uint32_t vm0 = tail->valid[kr][0], vm1 = tail->valid[kr][1];
        // P and dS of this chunk, packed to bf16 pairs in registers (8 keys at a time)
        uint32_t pw[32], dw[32];
#pragma unroll
        for (int qk = 0; qk < 8; ++qk) {
          uint32_t sv[8], dv[8];
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
              : "=r"(sv[0]), "=r"(sv[1]), "=r"(sv[2]), "=r"(sv[3]), "=r"(sv[4]), "=r"(sv[5]),
                "=r"(sv[6]), "=r"(sv[7])
              : "r"(tmem + lane_off + kColS + qk * 8)
              : "memory");
          asm volatile(
              "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
              : "=r"(dv[0]), "=r"(dv[1]), "=r"(dv[2]), "=r"(dv[3]), "=r"(dv[4]), "=r"(dv[5]),
                "=r"(dv[6]), "=r"(dv[7])
              : "r"(tmem + lane_off + kColDP + qk * 8)
              : "memory");
          tmem_ld_wait();
          const uint32_t vm = (qk < 4 ? vm0 : vm1) >> ((qk & 3) * 8);
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            const bool v0 = hv && ((vm >> j) & 1u), v1 = hv && ((vm >> (j + 1)) & 1u);
            const float p0 = v0 ? ex2b(fmaf(__uint_as_float(sv[j]), c2, -lse2)) : 0.f;
            const float p1 = v1 ? ex2b(fmaf(__uint_as_float(sv[j + 1]), c2, -lse2)) : 0.f;
            pw[qk * 4 + j / 2] = pack_bf16(p0, p1);
            dw[qk * 4 + j / 2] = pack_bf16(p0 * (__uint_as_float(dv[j]) - delta),
                                           p1 * (__uint_as_float(dv[j + 1]) - delta));
          }
        }
        // S / dP are in registers: the next chunk's S / dP may overwrite them
        tc_fence_before();
        mbar_arrive(&tail->sdp_free);
        // dS into its buffer once the chunk before the previous one has consumed it
        const int db = g & 1;
        if (g > 1 && !__all_sync(0xffffffffu, mbar_wait(&tail->ds_free[db], ((g >> 1) - 1) & 1,
                                                         abort_flag, p.err, kErrB))) {
          ok = false;
          break;
        }
        uint8_t* dsrow = dsrow0 + db * kQAtom;
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const uint32_t off = (static_cast<uint32_t>(cc) ^ sw) << 4;
          *reinterpret_cast<uint4*>(dsrow + off) =
              make_uint4(dw[cc * 4], dw[cc * 4 + 1], dw[cc * 4 + 2], dw[cc * 4 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&tail->ds_full[db]);
        // P once the previous chunk's dV^T has read it
        if (g > 0 && !__all_sync(0xffffffffu, mbar_wait(&tail->p_free, (g - 1) & 1, abort_flag,
                                                         p.err, kErrB))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int cc = 0; cc < 8; ++cc) {
          const uint32_t off = (static_cast<uint32_t>(cc) ^ sw) << 4;
          *reinterpret_cast<uint4*>(prow + off) =
              make_uint4(pw[cc * 4], pw[cc * 4 + 1], pw[cc * 4 + 2], pw[cc * 4 + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&tail->p_full);
        ++g;
      }
      if (!ok) break;
      // dQ of this row: scale * (sum over chunks of dS . K)
      if (!__all_sync(0xffffffffu, mbar_wait(&tail->dq_full, nrow & 1, abort_flag, p.err, kErrB))) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint4* qrow = reinterpret_cast<uint4*>(p.dQ + (row * H + hrow) * DQK);
#pragma unroll
      for (int d0 = 0; d0 < DQK; d0 += 32) {
        uint32_t v[32];
        tmem_ld_x32(tmem + lane_off + kColDQ + d0, v);
        tmem_ld_wait();
        if (hv) {
#pragma unroll
          for (int d = 0; d < 32; d += 8) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(v[d]) * p.scale, __uint_as_float(v[d + 1]) * p.scale);
            w.y = pack_bf16(__uint_as_float(v[d + 2]) * p.scale, __uint_as_float(v[d + 3]) * p.scale);
            w.z = pack_bf16(__uint_as_float(v[d + 4]) * p.scale, __uint_as_float(v[d + 5]) * p.scale);
            w.w = pack_bf16(__uint_as_float(v[d + 6]) * p.scale, __uint_as_float(v[d + 7]) * p.scale);
            qrow[(d0 + d) / 8] = w;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tail->dq_free);
    }
  } else {
    // ================================================================ drain
    // warp 4 + q + 4h owns TMEM lanes 32q..32q+31 (dims 32q.. of dK^T lo / dV^T and
    // 128+32q.. of dK^T hi for q < 2) and keys 32h..32h+31 of each chunk.
    const int dw_ = warp - 4;
    const int q = dw_ & 3, hk = dw_ >> 2;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    float* tile = reinterpret_cast<float*>(smem + kDrainOff + dw_ * kDrainTile);
    const int rr = lane >> 3, c4 = (lane & 7) * 4;
    int g = 0;
    bool ok = true;
    for (int i = blockIdx.x; ok && i < nrows; i += gridDim.x) {
      bool last = false;
      while (!last) {
        const int kr = g % kKeyRing;
        // the slot is not rewritten before this chunk has been drained
        if (!__all_sync(0xffffffffu, mbar_wait(&tail->keys_full[kr], (g / kKeyRing) & 1,
                                                abort_flag, p.err, kErrB))) {
          ok = false;
          break;
        }
        last = (tail->flags[kr] & 2) != 0;
        const int row = tail->row[kr];
        const int b = row / p.S;
        float* ws = p.ws + static_cast<long long>(b) * p.S * (DQK + DV);
        const int* keys = tail->key[kr];
        // regions in the order the tensor cores produce them: dK^T lo, dK^T hi (dims
        // 128-191: quarters 0-1), dV^T. Each 32-dim x 16-key block goes through a
        // shared tile so that a thread holds 4 consecutive dims of one key: one
        // 16-byte reduction per thread, 4 key rows x 128 contiguous bytes per warp
        // instruction.
#pragma unroll 1
        for (int ri = 0; ri < 3; ++ri) {
          const int reg = ri == 2 ? 0 : ri + 1;
          if (!__all_sync(0xffffffffu,
                          mbar_wait(&tail->dkv_full[reg], g & 1, abort_flag, p.err, kErrB))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (reg == 2 && q >= 2) {
            // dims 192-255 of the dK^T hi region do not exist
            tc_fence_before();
            mbar_arrive(&tail->dkv_free[reg]);
          } else {
            const uint32_t col = reg == 0 ? kColDV : (reg == 1 ? kColDKlo : kColDKhi);
            const int dim0 = (reg == 0 ? DQK : (reg == 1 ? 0 : 128)) + q * 32;
            const float sc = reg == 0 ? 1.f : p.scale;
            // both 16-key blocks of this warp into registers with one wait; the TMEM
            // region is then free for the next chunk's MMA while the reductions run
            // (the key indices too: once every region is released the ring slot may
            // be rewritten)
            uint32_t va[16], vb[16];
            tmem_ld_x16_b(tmem + lane_off + col + hk * 32, va);
            tmem_ld_x16_b(tmem + lane_off + col + hk * 32 + 16, vb);
            int kreg[2][4];
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll
              for (int i4 = 0; i4 < 4; ++i4) kreg[half][i4] = keys[hk * 32 + half * 16 + rr + 4 * i4];
            tmem_ld_wait();
            tc_fence_before();
            mbar_arrive(&tail->dkv_free[reg]);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                tile[j * kDrainPitch + lane] = __uint_as_float(half == 0 ? va[j] : vb[j]) * sc;
              __syncwarp();
#pragma unroll
              for (int i4 = 0; i4 < 4; ++i4) {
                const int r = rr + 4 * i4;
                const int key = kreg[half][i4];
                if (key >= 0) {
                  const float4 x = *reinterpret_cast<const float4*>(tile + r * kDrainPitch + c4);
                  atomicAdd(reinterpret_cast<float4*>(ws + static_cast<long long>(key) * (DQK + DV) +
                                                      dim0 + c4),
                            x);
                }
              }
              __syncwarp();
            }
          }
        }
        if (!ok) break;
        ++g;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

typedef CUresult (*EncodeTiledFnBwd)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                     const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                     const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                     CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_row_map(CUtensorMap* map, const void* base, long long rows, int cols) {
  static EncodeTiledFnBwd fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFnBwd>(ptr);
  }
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Any H <= 128: P and dS of the TMEM lanes >= H are zero, so those lanes add
// nothing to dK / dV, and their dQ is not stored.
bool attn_bwd_tc_supported(int H, int Dqk, int Dv, float scale) {
  return H >= 1 && H <= 128 && scale > 0.f && Dqk == 192 && Dv == 128;
}

// ws must be zeroed by the caller's stream before this runs.
int launch_attn_bwd_tc(const AttnParams& p, cudaStream_t stream) {
  const long long qrows = static_cast<long long>(p.B) * p.S * p.H;
  CUtensorMap mq, mdo;
  if (!make_row_map(&mq, p.Q, qrows, DQK) || !make_row_map(&mdo, p.dO, qrows, DV))
    return DSA_ERR_CUDA;
  const size_t smem = kTailOff + sizeof(BwdTail);
  if (cudaFuncSetAttribute(attn_bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long rows = static_cast<long long>(p.B) * p.S;
  const int grid = static_cast<int>(rows < sms ? rows : sms);
  attn_bwd_tc_kernel<<<grid, kThreads, smem, stream>>>(mq, mdo, p);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa
