// The indexer's auxiliary loss on the 5th-generation tensor cores.
//
// ("Implement QK attention head chunking for CSA": the indexer-loss target is the
// fp32 softmax of every head's attention scores over the valid tokens, summed over
// the heads and held constant; "Support Ring Attention with DeepSeek DSA Sparse
// Indexer", Loss Harvesting & Objective Injection: the loss joins the objective and
// its gradient reaches the indexer's query and key projections.)
//
// For query row t with selected slots j (0 <= s_j = idx[t,j] <= t):
//   pbar_j = (1/H) sum_h exp(scale Q[t,h].K[s_j] - LSE[t,h])      target (LSE from the
//                                                                   attention forward)
//   q_j    = exp(I[t,s_j] - logZ_t),  logZ_t = log sum_j exp(I[t,s_j])
//   L_t    = sum_j pbar_j (log pbar_j - log q_j)
//   dI_j   = g (q_j - pbar_j)                                       gradient of g sum_t L_t
// and, through I[t,s] = sum_h w[t,h] max(0, z_h), z_h = q_idx[t,h].k_idx[s]
// (derivative of max(0, z) at 0 taken as 0):
//   dw[t,h] = sum_j dI_j max(0, z_hj)
//   dq[t,h] = sum_j dI_j w[t,h] [z_hj > 0] k_idx[s_j]
//   dk[s_j] += sum_h dI_j w[t,h] [z_hj > 0] q_idx[t,h]
//
// Forward kernel. The keys of a chunk are the UMMA M dimension and the heads are N,
//   S^T[128 keys x H] = K_sel[128 x Dqk] . Q_t[H x Dqk]^T     (both operands K-major)
// so that each epilogue thread holds one key's logits for every head and sums the
// target over the heads inside the thread; no reduction crosses threads except the
// row's log-sum-exp of the index scores and the loss sum.
//
// Backward kernel. Per chunk of 128 keys, three products share two shared-memory tiles:
//   Z^T[128 keys x Hi]   = K_sel . q_t^T              K_sel and q_t K-major
//   dq^T[Di x Hi]       += K_sel^T . G                 both MN-major (the same tiles)
//   dk_rows[128 x Di]    = G . q_t                     G K-major, q_t MN-major
// where G[key, h] = dI w[t,h] [z > 0] is written by the epilogue as a bf16 tile. dq^T
// accumulates in TMEM over the row's chunks; each dk row is added to the output with
// 16-byte fp32 reductions; dw is reduced over the keys with a warp reduce-scatter.
//
// Both kernels: persistent CTA per SM, warp-specialised:
//   epilogue    forward: warps 0-7, two per TMEM lane quarter, each summing half of the
//               heads of a key; backward: warps 0-3 (one key, or one dimension of dq,
//               per thread)
//   issuer      forward: warp 8, backward: warp 4 - TMEM owner and single-thread UMMA
//               issuer
//   gather      forward: warps 9-12, backward: warps 5-8 - 16-byte cp.async of the
//               selected key rows into 128B-swizzled tiles, four keys per group so that
//               every copy instruction uses all 32 lanes; the row's Q (q_idx) tile
//               alongside its first chunk
//   drain       backward: warps 9-12 - the dk rows from TMEM into dk_idx (fp32
//               reductions), overlapping the epilogue's next chunk
// Every wait is bounded (the library's 2 s limit); a wait that runs out sets the
// CTA's abort flag and the error word, and every role then leaves its loops.

#include <cstdlib>

#include "dsa_common.cuh"
#include "dsa_internal.h"

namespace dsa {
namespace {

constexpr int kNK = 128;                 // keys per chunk (UMMA M)
constexpr int kGatherWarps = 4;
constexpr int kGatherThreads = 32 * kGatherWarps;
// forward: 8 epilogue warps, the issuer, 4 gather warps; backward: 4 epilogue warps, the
// issuer, 4 gather warps, 4 dk drain warps
constexpr int kFwdIssuer = 8, kFwdGather0 = 9, kFwdThreads = 416;
constexpr int kBwdIssuer = 4, kBwdGather0 = 5, kBwdDrain0 = 9, kBwdThreads = 416;
constexpr uint32_t kAtom = kNK * 128;    // [128 rows x 128 B] swizzle atom
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kErrFwd = DSA_STAGE_LOSS | DSA_DEVERR_TIMEOUT;
constexpr int kErrBwd = DSA_STAGE_LOSS_BWD | DSA_DEVERR_TIMEOUT;

static_assert(kNK == kGatherThreads, "one gather thread per key slot");

__device__ __forceinline__ void bar_gather() {
  asm volatile("bar.sync 1, %0;" ::"n"(kGatherThreads) : "memory");
}

// Named barrier of the gather threads that also agrees on whether to go on:
// thread 0 samples the abort flag before the barrier and everyone reads that one
// sample after it (two slots, so that a fast thread 0 cannot overwrite a verdict
// a slow thread has yet to read).
template <int W0>
__device__ __forceinline__ bool bar_gather_ok(int* okb, int& nb, volatile int* abort_flag) {
  if (threadIdx.x == 32 * W0) okb[nb & 1] = (*abort_flag == 0);
  bar_gather();
  const bool ok = reinterpret_cast<volatile int*>(okb)[nb & 1] != 0;
  ++nb;
  return ok;
}

__device__ __forceinline__ long long row_of(int i, int nrows) {
  return static_cast<long long>(nrows) - 1 - i;   // longest rows first
}

__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* err, int code) {
  const uint32_t a = smem_u32(bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      report_error(err, code);
      return;
    }
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// kind::f16 instruction descriptor with bf16 operands and an fp32 accumulator; each
// operand K-major or MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (a_mn ? (1u << 15) : 0u) |
         (b_mn ? (1u << 16) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// The gather threads' index list pass: one past the last slot that holds a key the
// row may attend to (0 <= s <= t), agreed by all gather threads. Returns false when
// the CTA is aborting.
template <int W0>
__device__ __forceinline__ bool row_kend(const int32_t* irow, int k, int t, int S, int gt,
                                         int lane, int gw, int* red, int* okb, int& nb,
                                         volatile int* abort_flag, int& kend) {
  int last = 0;
#pragma unroll 1
  for (int j0 = gt; j0 < k; j0 += 16 * kGatherThreads) {
    int sv[16];   // sixteen loads in flight per thread
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int j = j0 + u * kGatherThreads;
      sv[u] = j < k ? __ldg(irow + j) : -1;
    }
#pragma unroll
    for (int u = 0; u < 16; ++u)
      if (sv[u] >= 0 && sv[u] <= t && sv[u] < S) last = j0 + u * kGatherThreads + 1;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  if (lane == 0) red[gw] = last;
  if (!bar_gather_ok<W0>(okb, nb, abort_flag)) return false;
  kend = 0;
#pragma unroll
  for (int w2 = 0; w2 < kGatherWarps; ++w2) kend = max(kend, red[w2]);
  return true;
}

// key index in slot j of a row (the causal mask applied), -1 if none
__device__ __forceinline__ int slot_key(const int32_t* irow, int j, int kend, int t, int S) {
  if (j >= kend) return -1;
  const int s = __ldg(irow + j);
  return (s >= 0 && s <= t && s < S) ? s : -1;
}

// Copy the rows of 128 gathered keys (D bf16 each, D a multiple of 64) into a
// 128B-swizzled K-major tile [D/64 atoms][128 rows][128 B]. keys[] holds the 128
// key indices (-1: zero row); the gather threads take groups of four keys so that
// the 32 lanes of each copy instruction cover 4 x 128 contiguous bytes.
template <int D>
__device__ __forceinline__ void gather_rows(uint32_t stage, const int* keys,
                                            const __nv_bfloat16* base, int gw, int lane) {
  constexpr int PK = D / 8;   // 16-byte pieces per row
  constexpr int KI = PK / 8;  // copy instructions per group of 4 keys
#pragma unroll 1
  for (int grp = gw; grp < kNK / 4; grp += kGatherWarps) {
    const int4 kq = *reinterpret_cast<const int4*>(keys + grp * 4);
#pragma unroll
    for (int ii = 0; ii < KI; ++ii) {
      const int q = ii * 32 + lane, kig = q / PK, pc = q % PK;
      const int ks = kig == 0 ? kq.x : (kig == 1 ? kq.y : (kig == 2 ? kq.z : kq.w));
      const int key = grp * 4 + kig;
      const uint32_t dst = stage + (pc >> 3) * kAtom + key * 128 + (((pc & 7) ^ (key & 7)) << 4);
      cp_async_16(dst, base + static_cast<long long>(ks >= 0 ? ks : 0) * D + pc * 8,
                  ks >= 0 ? 16u : 0u);
    }
  }
}

// ===================================================================== forward

struct LossFwdParams {
  const __nv_bfloat16* Q;   // [B, S, H, DQK]
  const __nv_bfloat16* K;   // [B, S, DQK]
  const int32_t* idx;       // [B, S, k]
  const float* lse;         // [B, S, H]
  const float* scores;      // [B, S, ld]
  long long ld;
  int B, S, H, k;
  float c2;                 // scale * log2(e)
  float grad_scale;
  float* kl;                // [B, S], zeroed before the launch
  float* dI;                // [B, S, k]
  int* err;
};

constexpr int kFwdStages = 2;
constexpr int kFwdKeepChunks = 16;   // chunks whose scores the epilogue keeps from its pre-pass

template <int DQK>
struct LossFwdLayout {
  static constexpr int KA = DQK / 64;
  static constexpr uint32_t kStage = KA * kAtom;          // 128 keys x DQK
  static constexpr uint32_t kQOff = kFwdStages * kStage;  // Q tiles: [KA][128 rows][128 B]
  static constexpr uint32_t kQBuf = KA * kAtom;
  static constexpr uint32_t kTailOff = kQOff + 2 * kQBuf;
};

struct LossFwdTail {
  int first[kFwdStages], last[kFwdStages];
  __align__(16) int key[kFwdStages][kNK];   // read as int4 by gather_rows
  uint64_t kv_full[kFwdStages], kv_empty[kFwdStages];
  uint64_t s_full[kFwdStages], s_empty[kFwdStages];
  uint64_t e_full[kFwdStages];
  uint64_t q_empty[2];
  uint64_t lz_bar;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int okb[2];
  int red[kGatherWarps];
  __align__(16) float lse2[2][128];   // the row's LSE in log2 units, by row parity
  float lzm[2][8], lzl[2][8];         // per-warp partial log-sum-exp of the scores
  int lzk[2][8];                      // per-warp partial kend
  float ebuf[kFwdStages][128];        // the upper epilogue warps' partial head sums
  float sv[2][kFwdKeepChunks * 128];  // by row parity: the score (log2 units) at slot j of
                                      // the row's first kFwdKeepChunks chunks, NaN where
                                      // the slot holds no selected key
};

template <int DQK>
__global__ void __launch_bounds__(kFwdThreads, 1) loss_fwd_kernel(const LossFwdParams p) {
  using L = LossFwdLayout<DQK>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) report_error(p.err, DSA_STAGE_LOSS | DSA_DEVERR_MISALIGNED);
    return;
  }
  LossFwdTail* tail = reinterpret_cast<LossFwdTail*>(smem + L::kTailOff);
  volatile int* abort_flag = &tail->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrows = p.B * p.S;
  const int Hp = (p.H + 15) & ~15;   // UMMA N: heads rounded up to 16 (zero rows above H)

  if (threadIdx.x == 0) {
    for (int i = 0; i < kFwdStages; ++i) {
      // per gather thread: one arrive for its header write, one when its copies land
      mbar_init(&tail->kv_full[i], 2 * kGatherThreads);
      mbar_init(&tail->kv_empty[i], 1);
      mbar_init(&tail->s_full[i], 1);
      mbar_init(&tail->s_empty[i], 256);   // both epilogue warps of each lane quarter
      mbar_init(&tail->e_full[i], 128);    // the upper epilogue warps
    }
    mbar_init(&tail->q_empty[0], 1);
    mbar_init(&tail->q_empty[1], 1);
    mbar_init(&tail->lz_bar, 8);
    mbar_init(&tail->drain, 1);
    tail->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kFwdIssuer) {
    tmem_alloc(&tail->tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tail->tmem_base;

  if (warp >= kFwdGather0) {
    // ================================================================ gather
    const int gt = threadIdx.x - 32 * kFwdGather0;
    const int gw = warp - kFwdGather0;
    constexpr int PQ = DQK / 8;
    int g = 0, nb = 0, ri = 0;
    for (int i = blockIdx.x; i < nrows; i += gridDim.x, ++ri) {
      const long long row = row_of(i, nrows);
      const int b = static_cast<int>(row / p.S);
      const int t = static_cast<int>(row - static_cast<long long>(b) * p.S);
      const int32_t* irow = p.idx + row * p.k;
      int kend = 0;
      if (!row_kend<kFwdGather0>(irow, p.k, t, p.S, gt, lane, gw, tail->red, tail->okb, nb, abort_flag, kend))
        break;
      const int nch = kend > 0 ? (kend + kNK - 1) / kNK : 1;
      // the row's Q tile, once the MMAs of the row two back have read the buffer
      const int qb = ri & 1;
      mbar_wait(&tail->q_empty[qb], ((ri >> 1) & 1) ^ 1u, abort_flag, p.err, kErrFwd);
      if (!bar_gather_ok<kFwdGather0>(tail->okb, nb, abort_flag)) break;
      const uint32_t qbuf = smem_u32(smem + L::kQOff + qb * L::kQBuf);
      const __nv_bfloat16* qsrc = p.Q + row * p.H * DQK;
#pragma unroll 2
      for (int q = gt; q < Hp * PQ; q += kGatherThreads) {
        const int h = q / PQ, pc = q % PQ;
        const uint32_t dst = qbuf + (pc >> 3) * kAtom + h * 128 + (((pc & 7) ^ (h & 7)) << 4);
        cp_async_16(dst, qsrc + static_cast<long long>(h < p.H ? h : 0) * DQK + pc * 8,
                    h < p.H ? 16u : 0u);
      }
      bool stop = false;
      for (int c = 0; c < nch; ++c, ++g) {
        const int st = g % kFwdStages;
        const int s = slot_key(irow, c * kNK + gt, kend, t, p.S);
        mbar_wait(&tail->kv_empty[st], ((g / kFwdStages) & 1) ^ 1u, abort_flag, p.err, kErrFwd);
        tail->key[st][gt] = s;
        if (gt == 0) {
          tail->first[st] = c == 0;
          tail->last[st] = c == nch - 1;
        }
        if (!bar_gather_ok<kFwdGather0>(tail->okb, nb, abort_flag)) { stop = true; break; }
        mbar_arrive(&tail->kv_full[st]);   // releases the header writes
        gather_rows<DQK>(smem_u32(smem + st * L::kStage), tail->key[st],
                         p.K + static_cast<long long>(b) * p.S * DQK, gw, lane);
        // second arrival, by the copy hardware once this thread's copies (and the
        // row's Q pieces before them) have landed
        cp_async_mbar_arrive(&tail->kv_full[st]);
      }
      if (stop) break;
    }
    cp_async_wait<0>();
  } else if (warp == kFwdIssuer) {
    // ================================================================ UMMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, Hp, false, false);
      int g = 0, ri = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < nrows; i += gridDim.x, ++ri) {
        const int qb = ri & 1;
        const uint32_t qbase = smem_u32(smem + L::kQOff + qb * L::kQBuf);
        bool last = false;
        while (!last) {
          const int st = g % kFwdStages;
          const uint32_t par = (g / kFwdStages) & 1;
          if (!mbar_wait(&tail->kv_full[st], par, abort_flag, p.err, kErrFwd)) { ok = false; break; }
          last = tail->last[st] != 0;
          if (!mbar_wait(&tail->s_empty[st], par ^ 1u, abort_flag, p.err, kErrFwd)) { ok = false; break; }
          // the tiles were written by cp.async (generic proxy); the tensor cores read
          // them through the async proxy
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t kbase = smem_u32(smem + st * L::kStage);
#pragma unroll
          for (int kk = 0; kk < DQK / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
            umma_bf16(tmem + st * 128, umma_sdesc(kbase + off, 1024, kLayoutSw128),
                      umma_sdesc(qbase + off, 1024, kLayoutSw128), idesc, kk > 0 ? 1u : 0u);
          }
          umma_commit(&tail->s_full[st]);
          umma_commit(&tail->kv_empty[st]);
          if (last) umma_commit(&tail->q_empty[qb]);
          ++g;
        }
      }
      umma_commit(&tail->drain);
      drain_wait(&tail->drain, 0, p.err, kErrFwd);
    }
  } else {
    // ================================================================ epilogue
    // Warps w and w + 4 share TMEM lane quarter w % 4: the lower warp sums the heads of
    // the even 32-column blocks, the upper warp those of the odd blocks and hands its
    // partial sum over through ebuf; the lower warp finishes the slot (dI, the loss).
    const bool upper = warp >= 4;
    const int tid = threadIdx.x & 127;           // key slot of a chunk; TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int H = p.H;
    const float invH = 1.f / static_cast<float>(H);
    int g = 0, ri = 0;
    for (int i = blockIdx.x; i < nrows; i += gridDim.x, ++ri) {
      const long long row = row_of(i, nrows);
      const int t = static_cast<int>(row % p.S);
      const int par = ri & 1;
      const int32_t* irow = p.idx + row * p.k;
      // the row's scores by key (ld > 0), or the selected keys' scores by slot (ld == 0)
      const float* srow = p.scores + row * (p.ld > 0 ? p.ld : p.k);
      // the row's LSE (log2 units) and the log-sum-exp of its selected index scores:
      // the 256 epilogue threads read slots j = e + 256 u (sixteen loads in flight per
      // thread) and keep the scores of the first kFwdKeepChunks chunks in sv[par]
      const int et = threadIdx.x;   // 0..255
      if (et < H) tail->lse2[par][et] = __ldg(p.lse + row * H + et) * kLog2e;
      float m = -INFINITY, l = 0.f;
      int kl_end = 0;
      float* svr = tail->sv[par];
#pragma unroll 1
      for (int j0 = et; j0 < p.k; j0 += 16 * 256) {
        int sk[16];
        float vv[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int j = j0 + u * 256;
          sk[u] = j < p.k ? __ldg(irow + j) : -1;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int s = sk[u];
          if (s < -1 || s >= p.S) {
            report_error(p.err, DSA_STAGE_LOSS | DSA_DEVERR_BAD_INDEX);
            sk[u] = -1;
          } else if (s > t) {
            sk[u] = -1;
          }
          vv[u] = sk[u] >= 0 ? __ldg(srow + (p.ld > 0 ? sk[u] : j0 + u * 256)) * kLog2e : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int j = j0 + u * 256;
          if (j < kFwdKeepChunks * 128) svr[j] = sk[u] >= 0 ? vv[u] : __int_as_float(0x7fc00000);
          if (sk[u] < 0) continue;
          kl_end = j + 1;
          const float v = vv[u];
          if (v > m) {
            l = l * ex2(m - v) + 1.f;
            m = v;
          } else if (v > -INFINITY) {
            l += ex2(v - m);
          }
        }
      }
      // slots of the kept chunks past k read as "no key"
      for (int j = p.k + et; j < kFwdKeepChunks * 128; j += 256) svr[j] = __int_as_float(0x7fc00000);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float om = __shfl_xor_sync(0xffffffffu, m, o);
        const float ol = __shfl_xor_sync(0xffffffffu, l, o);
        kl_end = max(kl_end, __shfl_xor_sync(0xffffffffu, kl_end, o));
        const float mm = fmaxf(m, om);
        l = (m > -INFINITY ? l * ex2(m - mm) : 0.f) + (om > -INFINITY ? ol * ex2(om - mm) : 0.f);
        m = mm;
      }
      // every epilogue warp arrives, so that no warp starts row ri + 2, and rewrites this
      // row's slots, before all have left row ri
      __syncwarp();
      if (lane == 0) {
        tail->lzm[par][warp] = m;
        tail->lzl[par][warp] = l;
        tail->lzk[par][warp] = kl_end;
        mbar_arrive(&tail->lz_bar);
      }
      if (!__all_sync(0xffffffffu, mbar_wait(&tail->lz_bar, par, abort_flag, p.err, kErrFwd)))
        break;
      float M = -INFINITY;
      int kend = 0;
#pragma unroll
      for (int w2 = 0; w2 < 8; ++w2) {
        M = fmaxf(M, tail->lzm[par][w2]);
        kend = max(kend, tail->lzk[par][w2]);
      }
      float Lsum = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < 8; ++w2) {
        const float mw = tail->lzm[par][w2];
        if (mw > -INFINITY) Lsum += tail->lzl[par][w2] * ex2(mw - M);
      }
      const float logz2 = Lsum > 0.f ? M + log2f(Lsum) : -INFINITY;
      const int nch = kend > 0 ? (kend + kNK - 1) / kNK : 1;
      const float* lse2 = tail->lse2[par];
      float kl_acc = 0.f;
      bool ok = true;
      for (int c = 0; c < nch; ++c, ++g) {
        const int st = g % kFwdStages;
        const uint32_t ph = (g / kFwdStages) & 1;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tail->s_full[st], ph, abort_flag, p.err, kErrFwd))) {
          ok = false;
          break;
        }
        tc_fence_after();
        // sum over this warp's heads of exp2(S * c2 - LSE2[h])
        float e = 0.f;
#pragma unroll 1
        for (int cb = upper ? 32 : 0; cb < Hp; cb += 64) {
          uint32_t v[32];
          tmem_ld_x32(tmem + lane_off + st * 128 + cb, v);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 32; h += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(lse2 + cb + h);
            const float x0 = ex2(fmaf(__uint_as_float(v[h]), p.c2, -l4.x));
            const float x1 = ex2(fmaf(__uint_as_float(v[h + 1]), p.c2, -l4.y));
            const float x2 = ex2(fmaf(__uint_as_float(v[h + 2]), p.c2, -l4.z));
            const float x3 = ex2(fmaf(__uint_as_float(v[h + 3]), p.c2, -l4.w));
            if (cb + 32 <= H) {
              e += (x0 + x1) + (x2 + x3);
            } else {
              e += (cb + h < H ? x0 : 0.f) + (cb + h + 1 < H ? x1 : 0.f) +
                   (cb + h + 2 < H ? x2 : 0.f) + (cb + h + 3 < H ? x3 : 0.f);
            }
          }
        }
        if (upper) {
          tail->ebuf[st][tid] = e;
          tc_fence_before();
          mbar_arrive(&tail->e_full[st]);
          mbar_arrive(&tail->s_empty[st]);
          continue;
        }
        // the partner's half; the TMEM buffer (and with it ebuf[st]) is released only
        // after it has been read
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tail->e_full[st], ph, abort_flag, p.err, kErrFwd))) {
          ok = false;
          break;
        }
        e += tail->ebuf[st][tid];
        tc_fence_before();
        mbar_arrive(&tail->s_empty[st]);
        const int j = c * kNK + tid;
        // this slot's key and score: from the pre-pass, or read again past its reach
        bool valid;
        float v2 = 0.f;
        if (c < kFwdKeepChunks) {
          v2 = svr[j];
          valid = !isnan(v2);
        } else {
          const int s = slot_key(irow, j, kend, t, p.S);
          valid = s >= 0;
          if (valid) v2 = __ldg(srow + (p.ld > 0 ? s : j)) * kLog2e;
        }
        if (j < p.k) {
          float d = 0.f;
          if (valid) {
            const float pbar = e * invH;
            const float lq2 = v2 - logz2;   // log2 of the student
            d = p.grad_scale * (ex2(lq2) - pbar);
            if (pbar > 0.f) kl_acc += pbar * (log2f(pbar) - lq2);
          }
          p.dI[row * p.k + j] = d;
        }
      }
      if (!ok) break;
      if (!upper) {
        for (int j = nch * kNK + tid; j < p.k; j += 128) p.dI[row * p.k + j] = 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) kl_acc += __shfl_xor_sync(0xffffffffu, kl_acc, o);
        if (lane == 0 && kl_acc != 0.f) atomicAdd(p.kl + row, kl_acc * kLn2);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kFwdIssuer) tmem_dealloc(tmem, 256);
}

// ==================================================================== backward

// One step of a warp reduce-scatter: lanes with bit O set keep the upper HALF values
// and add their partner's, the others the lower HALF. Five steps from 64 values per
// lane leave lane l with the warp's sums of values 2l and 2l + 1.
template <int HALF, int O>
__device__ __forceinline__ void reduce_scatter_step(float* r, int lane) {
  const bool up = (lane & O) != 0;
#pragma unroll
  for (int h = 0; h < HALF; ++h) {
    const float send = up ? r[h] : r[h + HALF];
    const float keep = up ? r[h + HALF] : r[h];
    r[h] = keep + __shfl_xor_sync(0xffffffffu, send, O);
  }
}

struct LossBwdParams {
  const __nv_bfloat16* q;   // q_idx [B, S, HI, DI]
  const __nv_bfloat16* kx;  // k_idx [B, S, DI]
  const float* w;           // [B, S, HI]
  const int32_t* idx;       // [B, S, k]
  const float* dI;          // [B, S, k]
  int B, S, k;
  float* dq;                // [B, S, HI, DI]
  float* dk;                // [B, S, DI], zeroed before the launch
  float* dw;                // [B, S, HI]
  int* err;
};

constexpr int kBwdStages = 3;

template <int HI, int DI>
struct LossBwdLayout {
  static_assert(HI == 64 && DI == 128, "one 64-head G atom, M = DI = 128 for dq^T");
  static constexpr uint32_t kStage = (DI / 64) * kAtom;        // 128 keys x DI
  static constexpr uint32_t kQAtom = HI * 128;                 // [HI rows x 128 B]
  static constexpr uint32_t kQOff = kBwdStages * kStage;
  static constexpr uint32_t kQBuf = (DI / 64) * kQAtom;
  static constexpr uint32_t kGOff = kQOff + 2 * kQBuf;         // G tiles [128 keys x HI] bf16
  static constexpr uint32_t kGBuf = (HI / 64) * kAtom;
  static constexpr uint32_t kXOff = kGOff + 2 * kGBuf;          // dk transpose, 4 KB per warp
  static constexpr uint32_t kTailOff = kXOff + 4 * 4096;
  // TMEM columns
  static constexpr uint32_t kColZ = 0;              // 2 x HI
  static constexpr uint32_t kColDk = 2 * HI;        // 2 x DI
  static constexpr uint32_t kColDq = 2 * HI + 2 * DI;
  static_assert(kColDq + HI <= 512, "TMEM budget");
};

template <int HI>
struct LossBwdTail {
  int first[kBwdStages], last[kBwdStages];
  __align__(16) int key[kBwdStages][kNK];   // read as int4 by gather_rows
  float dval[kBwdStages][kNK];
  uint64_t kv_full[kBwdStages], kv_empty[kBwdStages];
  uint64_t z_full[2], z_empty[2];
  uint64_t g_full[2], g_empty[2];
  uint64_t dk_full[2], dk_empty[2];
  uint64_t dq_full, dq_free;
  uint64_t q_empty[2];
  uint64_t dw_bar;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int okb[2];
  int red[kGatherWarps];
  __align__(16) float wrow[2][HI];   // w[t, :] by row parity
  float dw_acc[2][HI];
  int dk_key[2][kNK];                // by chunk parity: each slot's key, -1 where nothing is added
  int dk_last[2];                    // by chunk parity: the row's last chunk
};

template <int HI, int DI>
__global__ void __launch_bounds__(kBwdThreads, 1) loss_bwd_kernel(const LossBwdParams p) {
  using L = LossBwdLayout<HI, DI>;
  using Tail = LossBwdTail<HI>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) report_error(p.err, DSA_STAGE_LOSS_BWD | DSA_DEVERR_MISALIGNED);
    return;
  }
  Tail* tail = reinterpret_cast<Tail*>(smem + L::kTailOff);
  volatile int* abort_flag = &tail->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nrows = p.B * p.S;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kBwdStages; ++i) {
      mbar_init(&tail->kv_full[i], 2 * kGatherThreads);
      mbar_init(&tail->kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tail->z_full[i], 1);
      mbar_init(&tail->z_empty[i], 128);
      mbar_init(&tail->g_full[i], 128);
      mbar_init(&tail->g_empty[i], 1);
      mbar_init(&tail->dk_full[i], 1);
      mbar_init(&tail->dk_empty[i], 128);
      mbar_init(&tail->q_empty[i], 1);
    }
    mbar_init(&tail->dq_full, 1);
    mbar_init(&tail->dq_free, 128);   // the epilogue warps; dk_empty counts the drain warps
    mbar_init(&tail->dw_bar, 4);
    mbar_init(&tail->drain, 1);
    tail->abort_flag = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < 2 * HI; i += blockDim.x) (&tail->dw_acc[0][0])[i] = 0.f;
  static_assert(kBwdDrain0 == kBwdGather0 + kGatherWarps && kBwdThreads == 32 * (kBwdDrain0 + 4),
                "backward roles: 4 epilogue, 1 issuer, 4 gather, 4 drain warps");
  if (warp == kBwdIssuer) {
    tmem_alloc(&tail->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tail->tmem_base;

  if (warp >= kBwdGather0 && warp < kBwdDrain0) {
    // ================================================================ gather
    const int gt = threadIdx.x - 32 * kBwdGather0;
    const int gw = warp - kBwdGather0;
    constexpr int PQ = DI / 8;
    int g = 0, nb = 0, ri = 0;
    for (int i = blockIdx.x; i < nrows; i += gridDim.x, ++ri) {
      const long long row = row_of(i, nrows);
      const int b = static_cast<int>(row / p.S);
      const int t = static_cast<int>(row - static_cast<long long>(b) * p.S);
      const int32_t* irow = p.idx + row * p.k;
      int kend = 0;
      if (!row_kend<kBwdGather0>(irow, p.k, t, p.S, gt, lane, gw, tail->red, tail->okb, nb, abort_flag, kend))
        break;
      const int nch = kend > 0 ? (kend + kNK - 1) / kNK : 1;
      const int qb = ri & 1;
      mbar_wait(&tail->q_empty[qb], ((ri >> 1) & 1) ^ 1u, abort_flag, p.err, kErrBwd);
      if (!bar_gather_ok<kBwdGather0>(tail->okb, nb, abort_flag)) break;
      // q_idx[t] as [DI/64 atoms][HI rows][128 B] and w[t, :]
      const uint32_t qbuf = smem_u32(smem + L::kQOff + qb * L::kQBuf);
      const __nv_bfloat16* qsrc = p.q + row * HI * DI;
#pragma unroll
      for (int q = gt; q < HI * PQ; q += kGatherThreads) {
        const int h = q / PQ, pc = q % PQ;
        cp_async_16(qbuf + (pc >> 3) * L::kQAtom + h * 128 + (((pc & 7) ^ (h & 7)) << 4),
                    qsrc + h * DI + pc * 8, 16u);
      }
      if (gt < HI) tail->wrow[qb][gt] = __ldg(p.w + row * HI + gt);
      bool stop = false;
      // this slot's key and dI one chunk ahead (two independent loads), so that their
      // latency overlaps the previous chunk's wait and copies
      const float* drow = p.dI + row * p.k;
      int s_next = slot_key(irow, gt, kend, t, p.S);
      float dv_next = gt < p.k ? __ldg(drow + gt) : 0.f;
      for (int c = 0; c < nch; ++c, ++g) {
        const int st = g % kBwdStages;
        const int s = s_next;
        const float dv = s >= 0 ? dv_next : 0.f;
        if (c + 1 < nch) {
          const int jn = (c + 1) * kNK + gt;
          s_next = slot_key(irow, jn, kend, t, p.S);
          dv_next = jn < p.k ? __ldg(drow + jn) : 0.f;
        }
        mbar_wait(&tail->kv_empty[st], ((g / kBwdStages) & 1) ^ 1u, abort_flag, p.err, kErrBwd);
        tail->key[st][gt] = s;
        tail->dval[st][gt] = dv;
        if (gt == 0) {
          tail->first[st] = c == 0;
          tail->last[st] = c == nch - 1;
        }
        if (!bar_gather_ok<kBwdGather0>(tail->okb, nb, abort_flag)) { stop = true; break; }
        mbar_arrive(&tail->kv_full[st]);   // releases the header (and w row) writes
        gather_rows<DI>(smem_u32(smem + st * L::kStage), tail->key[st],
                        p.kx + static_cast<long long>(b) * p.S * DI, gw, lane);
        cp_async_mbar_arrive(&tail->kv_full[st]);
      }
      if (stop) break;
    }
    cp_async_wait<0>();
  } else if (warp == kBwdIssuer) {
    // ================================================================ UMMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_z = idesc_bf16(128, HI, false, false);    // Z^T = K . q^T
      constexpr uint32_t idesc_dq = idesc_bf16(DI, HI, true, true);      // dq^T += K^T . G
      constexpr uint32_t idesc_dk = idesc_bf16(128, DI, false, true);    // dk = G . q
      int g = 0, ri = 0, rq = 0;
      bool ok = true;
      int pend = -1, pend_first = 0, pend_last = 0, pend_qb = 0;
      // dq and dk products of chunk gp, once its G tile is in shared memory
      auto grads = [&](int gp, int first, int last, int qb) -> bool {
        const int pst = gp % kBwdStages, gb = gp & 1;
        const uint32_t ph = (gp >> 1) & 1;
        if (!mbar_wait(&tail->g_full[gb], ph, abort_flag, p.err, kErrBwd)) return false;
        if (!mbar_wait(&tail->dk_empty[gb], ph ^ 1u, abort_flag, p.err, kErrBwd)) return false;
        if (first) {
          if (!mbar_wait(&tail->dq_free, (rq & 1) ^ 1u, abort_flag, p.err, kErrBwd)) return false;
          ++rq;
        }
        // G was written by the epilogue's st.shared (fenced to the async proxy there)
        tc_fence_after();
        const uint32_t kbase = smem_u32(smem + pst * L::kStage);
        const uint32_t gbase = smem_u32(smem + L::kGOff + gb * L::kGBuf);
        const uint32_t qbase = smem_u32(smem + L::kQOff + qb * L::kQBuf);
#pragma unroll
        for (int ks = 0; ks < kNK / 16; ++ks)
          umma_bf16(tmem + L::kColDq,
                    umma_sdesc_lbo(kbase + ks * 2048, kAtom, 1024, kLayoutSw128),
                    umma_sdesc_lbo(gbase + ks * 2048, kAtom, 1024, kLayoutSw128), idesc_dq,
                    (first && ks == 0) ? 0u : 1u);
#pragma unroll
        for (int kk = 0; kk < HI / 16; ++kk)
          umma_bf16(tmem + L::kColDk + gb * DI,
                    umma_sdesc(gbase + (kk >> 2) * kAtom + (kk & 3) * 32, 1024, kLayoutSw128),
                    umma_sdesc_lbo(qbase + kk * 2048, L::kQAtom, 1024, kLayoutSw128), idesc_dk,
                    kk > 0 ? 1u : 0u);
        umma_commit(&tail->dk_full[gb]);
        umma_commit(&tail->kv_empty[pst]);
        umma_commit(&tail->g_empty[gb]);
        if (last) {
          umma_commit(&tail->dq_full);
          umma_commit(&tail->q_empty[qb]);
        }
        return true;
      };
      for (int i = blockIdx.x; ok && i < nrows; i += gridDim.x, ++ri) {
        const int qb = ri & 1;
        const uint32_t qbase = smem_u32(smem + L::kQOff + qb * L::kQBuf);
        bool last = false;
        while (!last) {
          const int st = g % kBwdStages, zb = g & 1;
          if (!mbar_wait(&tail->kv_full[st], (g / kBwdStages) & 1, abort_flag, p.err, kErrBwd)) {
            ok = false;
            break;
          }
          last = tail->last[st] != 0;
          const int first = tail->first[st];
          if (!mbar_wait(&tail->z_empty[zb], ((g >> 1) & 1) ^ 1u, abort_flag, p.err, kErrBwd)) {
            ok = false;
            break;
          }
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t kbase = smem_u32(smem + st * L::kStage);
#pragma unroll
          for (int kk = 0; kk < DI / 16; ++kk) {
            umma_bf16(tmem + L::kColZ + zb * HI,
                      umma_sdesc(kbase + (kk >> 2) * kAtom + (kk & 3) * 32, 1024, kLayoutSw128),
                      umma_sdesc(qbase + (kk >> 2) * L::kQAtom + (kk & 3) * 32, 1024,
                                 kLayoutSw128),
                      idesc_z, kk > 0 ? 1u : 0u);
          }
          umma_commit(&tail->z_full[zb]);
          if (pend >= 0) {
            if (!grads(pend, pend_first, pend_last, pend_qb)) { ok = false; break; }
            pend = -1;
          }
          if (last) {
            // the row's last chunk: its products right away, so that dq is complete
            if (!grads(g, first, 1, qb)) { ok = false; break; }
          } else {
            pend = g;
            pend_first = first;
            pend_last = 0;
            pend_qb = qb;
          }
          ++g;
        }
      }
      umma_commit(&tail->drain);
      drain_wait(&tail->drain, 0, p.err, kErrBwd);
    }
  } else if (warp >= kBwdDrain0) {
    // ================================================================ dk drain
    // Thread tq holds key slot tq's dk row in TMEM (lane quarter warp % 4). The warp passes
    // 32 columns of its 32 keys through a swizzled shared tile so that each quarter-warp adds
    // one key's 128 contiguous bytes per reduction instruction.
    const int quarter = warp & 3;
    const int tq = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t xt = smem_u32(smem + L::kXOff) + quarter * 4096;
    const int sub = lane >> 3, pc = lane & 7;
    int g = 0;
    bool ok = true;
    for (int i = blockIdx.x; ok && i < nrows; i += gridDim.x) {
      const long long row = row_of(i, nrows);
      const long long kvbase = row / p.S * p.S;
      bool last = false;
      while (!last) {
        const int db = g & 1;
        const uint32_t ph = (g >> 1) & 1;
        // the epilogue's handover (g_full) and the dk products (dk_full) of chunk g
        if (!__all_sync(0xffffffffu, mbar_wait(&tail->g_full[db], ph, abort_flag, p.err,
                                               kErrBwd)) ||
            !__all_sync(0xffffffffu, mbar_wait(&tail->dk_full[db], ph, abort_flag, p.err,
                                               kErrBwd))) {
          ok = false;
          break;
        }
        tc_fence_after();
        last = tail->dk_last[db] != 0;
        const int s = tail->dk_key[db][tq];
#pragma unroll 1
        for (int c0 = 0; c0 < DI; c0 += 32) {
          uint32_t v[32];
          tmem_ld_x32(tmem + lane_off + L::kColDk + db * DI + c0, v);
          tmem_ld_wait();
          __syncwarp();
#pragma unroll
          for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             xt + lane * 128 + ((c ^ (lane & 7)) << 4)),
                         "r"(v[4 * c]), "r"(v[4 * c + 1]), "r"(v[4 * c + 2]), "r"(v[4 * c + 3])
                         : "memory");
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int kr = 4 * u + sub;   // key row of this quarter-warp
            const int sk = __shfl_sync(0xffffffffu, s, kr);
            float4 x;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(x.x), "=f"(x.y), "=f"(x.z), "=f"(x.w)
                         : "r"(xt + kr * 128 + ((pc ^ (kr & 7)) << 4)));
            if (sk >= 0) {
              float* dst = p.dk + (kvbase + sk) * DI + c0 + pc * 4;
              asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(x.x),
                           "f"(x.y), "f"(x.z), "f"(x.w)
                           : "memory");
            }
          }
        }
        tc_fence_before();
        mbar_arrive(&tail->dk_empty[db]);
        ++g;
      }
    }
  } else {
    // ================================================================ epilogue
    const int tid = threadIdx.x;   // key slot of a chunk (Z, G); dimension of dq
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    int g = 0, ri = 0;
    bool ok = true;
    for (int i = blockIdx.x; i < nrows; i += gridDim.x, ++ri) {
      const long long row = row_of(i, nrows);
      const int par = ri & 1;
      bool last = false;
      while (!last) {
        const int st = g % kBwdStages, zb = g & 1;
        const uint32_t ph = (g >> 1) & 1;
        // the gather's header for this chunk (key, dI, last) and the row's w
        if (!__all_sync(0xffffffffu, mbar_wait(&tail->kv_full[st], (g / kBwdStages) & 1,
                                               abort_flag, p.err, kErrBwd))) {
          ok = false;
          break;
        }
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tail->z_full[zb], ph, abort_flag, p.err, kErrBwd))) {
          ok = false;
          break;
        }
        tc_fence_after();
        last = tail->last[st] != 0;
        const int s = tail->key[st][tid];
        const float d = tail->dval[st][tid];
        uint32_t z[HI];
#pragma unroll
        for (int c0 = 0; c0 < HI; c0 += 32)
          tmem_ld_x32(tmem + lane_off + L::kColZ + zb * HI + c0,
                      *reinterpret_cast<uint32_t(*)[32]>(z + c0));
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&tail->z_empty[zb]);
        // G = d w [z > 0] as bf16 pairs; z becomes d max(z, 0) (the dw terms)
        const float* wr = tail->wrow[par];
        uint32_t gp2[HI / 2];
#pragma unroll
        for (int h = 0; h < HI; h += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(wr + h);
          const float z0 = __uint_as_float(z[h]), z1 = __uint_as_float(z[h + 1]);
          const float z2 = __uint_as_float(z[h + 2]), z3 = __uint_as_float(z[h + 3]);
          gp2[h / 2] = pack_bf16(z0 > 0.f ? d * w4.x : 0.f, z1 > 0.f ? d * w4.y : 0.f);
          gp2[h / 2 + 1] = pack_bf16(z2 > 0.f ? d * w4.z : 0.f, z3 > 0.f ? d * w4.w : 0.f);
          z[h] = __float_as_uint(d * fmaxf(z0, 0.f));
          z[h + 1] = __float_as_uint(d * fmaxf(z1, 0.f));
          z[h + 2] = __float_as_uint(d * fmaxf(z2, 0.f));
          z[h + 3] = __float_as_uint(d * fmaxf(z3, 0.f));
        }
        // G row into its 128B-swizzled tile, once the products two chunks back are done
        const int gb = g & 1;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tail->g_empty[gb], ph ^ 1u, abort_flag, p.err, kErrBwd))) {
          ok = false;
          break;
        }
        // hand this chunk's keys to the drain warps, once they have drained the chunk that
        // used the buffer two chunks back (dk_key / dk_last are released by g_full)
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&tail->dk_empty[gb], ph ^ 1u, abort_flag, p.err, kErrBwd))) {
          ok = false;
          break;
        }
        tail->dk_key[gb][tid] = (s >= 0 && d != 0.f) ? s : -1;
        if (tid == 0) tail->dk_last[gb] = last ? 1 : 0;
        const uint32_t grow = smem_u32(smem + L::kGOff + gb * L::kGBuf) + tid * 128;
#pragma unroll
        for (int a = 0; a < HI / 64; ++a) {
#pragma unroll
          for (int c16 = 0; c16 < 8; ++c16) {
            const int wd = a * 32 + c16 * 4;
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             grow + a * kAtom + ((c16 ^ (tid & 7)) << 4)),
                         "r"(gp2[wd]), "r"(gp2[wd + 1]), "r"(gp2[wd + 2]), "r"(gp2[wd + 3])
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(&tail->g_full[gb]);
        // dw: reduce the 32 keys of the warp, ending with heads 2*lane and 2*lane + 1
        float r[HI];
#pragma unroll
        for (int h = 0; h < HI; ++h) r[h] = __uint_as_float(z[h]);
        reduce_scatter_step<32, 16>(r, lane);
        reduce_scatter_step<16, 8>(r, lane);
        reduce_scatter_step<8, 4>(r, lane);
        reduce_scatter_step<4, 2>(r, lane);
        reduce_scatter_step<2, 1>(r, lane);
        atomicAdd(&tail->dw_acc[par][2 * lane], r[0]);
        atomicAdd(&tail->dw_acc[par][2 * lane + 1], r[1]);
        ++g;
      }
      if (!ok) break;
      // dq^T of the row: thread tid holds dimension tid of every head
      if (!__all_sync(0xffffffffu, mbar_wait(&tail->dq_full, par, abort_flag, p.err, kErrBwd)))
        break;
      tc_fence_after();
      float* dqrow = p.dq + row * HI * DI + tid;
#pragma unroll
      for (int c0 = 0; c0 < HI; c0 += 32) {
        uint32_t v[32];
        tmem_ld_x32(tmem + lane_off + L::kColDq + c0, v);
        tmem_ld_wait();
#pragma unroll
        for (int h = 0; h < 32; ++h) dqrow[(c0 + h) * DI] = __uint_as_float(v[h]);
      }
      tc_fence_before();
      mbar_arrive(&tail->dq_free);
      // dw of the row once every warp has added its part
      __syncwarp();
      if (lane == 0) mbar_arrive(&tail->dw_bar);
      if (!__all_sync(0xffffffffu, mbar_wait(&tail->dw_bar, par, abort_flag, p.err, kErrBwd)))
        break;
      if (tid < HI) {
        p.dw[row * HI + tid] = tail->dw_acc[par][tid];
        tail->dw_acc[par][tid] = 0.f;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kBwdIssuer) tmem_dealloc(tmem, 512);
}

int sm_count() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms > 0 ? sms : 1;
}

template <int DQK>
int launch_fwd(const LossFwdParams& p, cudaStream_t stream) {
  using L = LossFwdLayout<DQK>;
  const size_t smem = L::kTailOff + sizeof(LossFwdTail);
  auto kern = loss_fwd_kernel<DQK>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  const long long rows = static_cast<long long>(p.B) * p.S;
  const int sms = sm_count();
  kern<<<static_cast<int>(rows < sms ? rows : sms), kFwdThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

template <int HI, int DI>
int launch_bwd(const LossBwdParams& p, cudaStream_t stream) {
  using L = LossBwdLayout<HI, DI>;
  const size_t smem = L::kTailOff + sizeof(LossBwdTail<HI>);
  auto kern = loss_bwd_kernel<HI, DI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return DSA_ERR_CUDA;
  const long long rows = static_cast<long long>(p.B) * p.S;
  const int sms = sm_count();
  kern<<<static_cast<int>(rows < sms ? rows : sms), kBwdThreads, smem, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

bool indexer_loss_supported(int H, int Dqk, float scale) {
  return H >= 1 && H <= 128 && scale > 0.f && (Dqk == 128 || Dqk == 192);
}

bool indexer_loss_bwd_supported(int Hi, int Di) { return Hi == 64 && Di == 128; }

int launch_indexer_loss(const void* Q, const void* K, const int32_t* idx, const float* lse,
                        const float* scores, int64_t ld, int B, int S, int H, int Dqk, int k,
                        float scale, float grad_scale, float* kl, float* dI,
                        cudaStream_t stream) {
  if (cudaMemsetAsync(kl, 0, sizeof(float) * static_cast<size_t>(B) * S, stream) != cudaSuccess)
    return DSA_ERR_CUDA;
  LossFwdParams p;
  p.Q = static_cast<const __nv_bfloat16*>(Q);
  p.K = static_cast<const __nv_bfloat16*>(K);
  p.idx = idx;
  p.lse = lse;
  p.scores = scores;
  p.ld = ld;
  p.B = B;
  p.S = S;
  p.H = H;
  p.k = k;
  p.c2 = scale * kLog2e;
  p.grad_scale = grad_scale;
  p.kl = kl;
  p.dI = dI;
  p.err = device_error_word();
  if (Dqk == 192) return launch_fwd<192>(p, stream);
  if (Dqk == 128) return launch_fwd<128>(p, stream);
  return DSA_ERR_UNSUPPORTED;
}

int launch_indexer_loss_bwd(const void* q_idx, const void* k_idx, const float* w,
                            const int32_t* idx, const float* dI, int B, int S, int Hi, int Di,
                            int k, float* dq, float* dk, float* dw, cudaStream_t stream) {
  if (cudaMemsetAsync(dk, 0, sizeof(float) * static_cast<size_t>(B) * S * Di, stream) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  LossBwdParams p;
  p.q = static_cast<const __nv_bfloat16*>(q_idx);
  p.kx = static_cast<const __nv_bfloat16*>(k_idx);
  p.w = w;
  p.idx = idx;
  p.dI = dI;
  p.B = B;
  p.S = S;
  p.k = k;
  p.dq = dq;
  p.dk = dk;
  p.dw = dw;
  p.err = device_error_word();
  if (Hi == 64 && Di == 128) return launch_bwd<64, 128>(p, stream);
  return DSA_ERR_UNSUPPORTED;
}

}  // namespace dsa
