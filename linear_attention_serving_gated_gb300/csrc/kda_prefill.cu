// kda_prefill.cu -- chunked varlen prefill from an indexed state pool.
//
// Contract: chunk_kda in "PR #35197 report: fix(kernel) Fix Helion small-token
// prefill bug" (implementation steps 1-2, key source snippet of
// kda_prefill.py): an indexed initial-state pool is required, gate/beta rows
// past the q token count are CUDA-graph bucket padding and are never read, a
// T = 1 prefill takes the same path as any other length, and varlen
// sequences are delimited by cu_seqlens.  The raw-beta flag is forwarded as
// in "[KDA] Support Helion MTP verification and harden prefill, decode"
// (sglang PR #42857, Modifications).
//
// Method: the 64-token chunk form of the gated delta rule.  For a chunk of L
// tokens starting from state S0 (K x V), with Gam the inclusive cumulative
// log-decay per key channel:
//   A[t,i] = beta_t sum_c k_t[c] k_i[c] e^{Gam_t[c]-Gam_i[c]}  (i < t)
//   P[t,i] =        sum_c q_t[c] k_i[c] e^{Gam_t[c]-Gam_i[c]}  (i <= t)
//   W      = (I+A)^-1 Diag(beta) Ktil,  Ktil_t = k_t e^{Gam_t}
//   Util   = (I+A)^-1 Diag(beta) V
//   U      = Util - W S0
//   O      = scale (Qtil S0 + P U),     Qtil_t = q_t e^{Gam_t}
//   S_L    = Diag(e^{Gam_L}) S0 + Khat^T U,  Khat_i = k_i e^{Gam_L - Gam_i}
// Rows past the end of a sequence are q = k = v = 0, beta = 0, g = 0, which
// leave every quantity above unchanged.
//
// Decay factors inside A and P are split at a reference token r, the LAST
// token of each 16-token block of i: e^{Gam_t-Gam_i} = e^{Gam_t-Gam_r} e^{Gam_r-Gam_i}.
// The right factor is <= 1 for every i of the block.  The left factor is <= 1
// for t >= r and at most e^{15 |g|min} for the block's own earlier rows, which
// stays inside FP32 for per-token log-decays >= -5.8 (the bounded gate at
// lower bound -5 is inside that).  A left factor that underflows can only
// drop terms that are smaller still.
//
// This file holds two kernels, both plain FP32 on the CUDA cores:
//   chunk_transform_kernel  one CTA per (chunk, head), all chunks in parallel:
//                           fold, cumulative decay, A, P, (I+A)^-1 by column
//                           forward substitution, W, Util, Qtil, Khat, gamma,
//                           written to the workspace.
//   state_pass_kernel       one CTA per (sequence, head, 16 value columns),
//                           sequential over the sequence's chunks: gathers S0
//                           from the pool, applies U, O and the state update,
//                           writes o, optional chunk-start states and scatters
//                           the final state back.
#include "kda_host.h"

namespace kda {
namespace {

constexpr int kChunk = 64;
constexpr int kLd = 132;  // padded row stride (floats) of 64 x 128 tiles in shared memory
constexpr int kLdT = 65;  // padded row stride of 64 x 64 tiles

// Workspace record of one (chunk, head), in floats.
constexpr int kOffW = 0;
constexpr int kOffU = kOffW + kChunk * kHeadDim;
constexpr int kOffQ = kOffU + kChunk * kHeadDim;
constexpr int kOffKh = kOffQ + kChunk * kHeadDim;
constexpr int kOffP = kOffKh + kChunk * kHeadDim;
constexpr int kOffGam = kOffP + kChunk * kChunk;
constexpr int kRec = kOffGam + kHeadDim;

struct PrefillArgs {
  GateArgs gate;
  int H, HV;
  const kda_bf16 *q, *k, *v, *g, *beta;
  float* pool;
  int pool_slots;
  const int32_t* state_idx;
  const int32_t* cu_seqlens;  // nullptr: fixed layout
  int num_seqs;
  int64_t total_tokens;
  kda_bf16* o;
  float* intermediate;
  float* ws;
  int32_t* err_flag;
};

__device__ __forceinline__ int64_t seq_begin(const PrefillArgs& a, int n) {
  return a.cu_seqlens ? (int64_t)a.cu_seqlens[n] : a.total_tokens / a.num_seqs * n;
}

// Checks cu_seqlens (0 .. total_tokens, non-decreasing).  One thread.
__device__ bool seqlens_valid(const PrefillArgs& a) {
  if (!a.cu_seqlens) return true;
  if (a.cu_seqlens[0] != 0 || a.cu_seqlens[a.num_seqs] != a.total_tokens) return false;
  for (int n = 0; n < a.num_seqs; ++n)
    if (a.cu_seqlens[n + 1] < a.cu_seqlens[n]) return false;
  return true;
}

struct ChunkLoc {
  int n;        // sequence, -1 if the chunk id is past the last chunk
  int64_t t0;   // first token of the chunk
  int len;      // tokens in the chunk (1..64)
};

// Maps a global chunk id (sequence-major) to its sequence and token range.
__device__ ChunkLoc locate_chunk(const PrefillArgs& a, int64_t cid) {
  int64_t base = 0;
  for (int n = 0; n < a.num_seqs; ++n) {
    const int64_t b = seq_begin(a, n), e = seq_begin(a, n + 1);
    const int64_t nch = (e - b + kChunk - 1) / kChunk;
    if (cid < base + nch) {
      const int64_t t0 = b + (cid - base) * kChunk;
      return ChunkLoc{n, t0, (int)(e - t0 < kChunk ? e - t0 : kChunk)};
    }
    base += nch;
  }
  return ChunkLoc{-1, 0, 0};
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int m = 16; m; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

__device__ __forceinline__ float4& f4(float* p) { return *reinterpret_cast<float4*>(p); }

// ---------------------------------------------------------------------------
// Per-chunk transform (all chunks of all sequences in parallel).

__global__ void __launch_bounds__(256) chunk_transform_kernel(const PrefillArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* KQ = sm;                    // k-hat      [64][kLd]
  float* QQ = KQ + kChunk * kLd;     // q-hat      [64][kLd]
  float* GM = QQ + kChunk * kLd;     // Gam        [64][kLd]
  float* L1 = GM + kChunk * kLd;     // Lk, later beta*Ktil, beta*V
  float* L2 = L1 + kChunk * kLd;     // Lq, later (I+A)^-1 [64][kLdT]
  float* R = L2 + kChunk * kLd;      // right factor [16][kLd]
  float* Am = R + 16 * kLd;          // A [64][kLdT]
  float* Pm = Am + kChunk * kLdT;    // P [64][kLdT]
  float* bt = Pm + kChunk * kLdT;    // beta [64]
  __shared__ ChunkLoc loc;
  __shared__ int skip;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.y;
  const int64_t cid = blockIdx.x;
  if (tid == 0) {
    skip = 0;
    if (!seqlens_valid(a)) {
      skip = 1;
      if (cid == 0 && h == 0) set_error(a.err_flag, KDA_DEVERR_SEQLENS);
    } else {
      loc = locate_chunk(a, cid);
      if (loc.n < 0) {
        skip = 1;
      } else {
        const int slot = a.state_idx[loc.n];
        if (slot < 0 || slot >= a.pool_slots) skip = 1;  // padding / rejected sequence
      }
    }
  }
  __syncthreads();
  if (skip) return;
  const int len = loc.len;
  const int64_t t0 = loc.t0;
  const GateArgs& ga = a.gate;
  const int H = a.H, HV = a.HV, K = kHeadDim;

  // 1. fold: one warp per token, 4 channels per lane.
  {
    const int c = lane * 4;
    const float exp_alog = ga.A_log ? expf(ga.A_log[h]) : 0.f;
    const float4 bias = ga.dt_bias ? *reinterpret_cast<const float4*>(ga.dt_bias + h * K + c)
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
    for (int t = warp; t < kChunk; t += 8) {
      float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f), k4 = q4, g4 = q4;
      if (t < len) {
        const int64_t tok = t0 + t;
        q4 = load_bf16x4(a.q + (tok * H + h) * K + c);
        k4 = load_bf16x4(a.k + (tok * H + h) * K + c);
        const float4 a4 = load_bf16x4(a.g + (tok * HV + h) * K + c);
        if (ga.use_qk_l2norm) {
          const float rq = rsqrtf(warp_sum(dot4(q4, q4)) + kNormEps);
          const float rk = rsqrtf(warp_sum(dot4(k4, k4)) + kNormEps);
          q4 = make_float4(q4.x * rq, q4.y * rq, q4.z * rq, q4.w * rq);
          k4 = make_float4(k4.x * rk, k4.y * rk, k4.z * rk, k4.w * rk);
        }
        g4 = make_float4(gate_log_decay(ga, a4.x, exp_alog, bias.x),
                         gate_log_decay(ga, a4.y, exp_alog, bias.y),
                         gate_log_decay(ga, a4.z, exp_alog, bias.z),
                         gate_log_decay(ga, a4.w, exp_alog, bias.w));
        if (lane == 0) bt[t] = fold_beta(ga, bf16_bits_to_float(a.beta[tok * HV + h]));
      } else if (lane == 0) {
        bt[t] = 0.f;
      }
      f4(QQ + t * kLd + c) = q4;
      f4(KQ + t * kLd + c) = k4;
      f4(GM + t * kLd + c) = g4;
    }
  }
  for (int i = tid; i < kChunk * kLdT; i += blockDim.x) {
    Am[i] = 0.f;
    Pm[i] = 0.f;
  }
  __syncthreads();

  // 2. inclusive cumulative log-decay per channel
  if (tid < K) {
    float run = 0.f;
    for (int t = 0; t < kChunk; ++t) {
      run += GM[t * kLd + tid];
      GM[t * kLd + tid] = run;
    }
  }
  __syncthreads();

  // 3. A and P, one 16-token block of i at a time, reference r = block end.
  for (int ib = 0; ib < kChunk / 16; ++ib) {
    const int b0 = ib * 16, r = b0 + 15;
    for (int idx = tid; idx < (kChunk - b0) * (K / 4); idx += blockDim.x) {
      const int t = b0 + idx / (K / 4), c = (idx % (K / 4)) * 4;
      const float4 gt = f4(GM + t * kLd + c), gr = f4(GM + r * kLd + c);
      const float4 kk = f4(KQ + t * kLd + c), qq = f4(QQ + t * kLd + c);
      const float4 e = make_float4(expf(gt.x - gr.x), expf(gt.y - gr.y), expf(gt.z - gr.z),
                                   expf(gt.w - gr.w));
      f4(L1 + t * kLd + c) = make_float4(kk.x * e.x, kk.y * e.y, kk.z * e.z, kk.w * e.w);
      f4(L2 + t * kLd + c) = make_float4(qq.x * e.x, qq.y * e.y, qq.z * e.z, qq.w * e.w);
      if (t <= r) {  // right factor of token t as i: k_i e^{Gam_r - Gam_i}
        const float4 f = make_float4(expf(gr.x - gt.x), expf(gr.y - gt.y), expf(gr.z - gt.z),
                                     expf(gr.w - gt.w));
        f4(R + (t - b0) * kLd + c) = make_float4(kk.x * f.x, kk.y * f.y, kk.z * f.z, kk.w * f.w);
      }
    }
    __syncthreads();
    for (int idx = tid; idx < (kChunk - b0) * 16; idx += blockDim.x) {
      const int t = b0 + idx / 16, i = b0 + idx % 16;
      if (i > t) continue;
      float sa = 0.f, sp = 0.f;
      const float* lk = L1 + t * kLd;
      const float* lq = L2 + t * kLd;
      const float* rr = R + (i - b0) * kLd;
#pragma unroll 8
      for (int c = 0; c < K; c += 4) {
        const float4 rv = f4(const_cast<float*>(rr) + c);
        sa += dot4(f4(const_cast<float*>(lk) + c), rv);
        sp += dot4(f4(const_cast<float*>(lq) + c), rv);
      }
      if (i < t) Am[t * kLdT + i] = bt[t] * sa;
      Pm[t * kLdT + i] = sp;
    }
    __syncthreads();
  }

  // 4. (I + A)^-1 by forward substitution, one column per thread.
  float* Ti = L2;
  if (tid < kChunk) {
    const int j = tid;
    for (int t = 0; t < kChunk; ++t) {
      float x;
      if (t < j) {
        x = 0.f;
      } else if (t == j) {
        x = 1.f;
      } else {
        x = 0.f;
        for (int i = j; i < t; ++i) x -= Am[t * kLdT + i] * Ti[i * kLdT + j];
      }
      Ti[t * kLdT + j] = x;
    }
  }
  // beta_i Ktil_i = beta_i k_i e^{Gam_i}
  for (int idx = tid; idx < kChunk * (K / 4); idx += blockDim.x) {
    const int i = idx / (K / 4), c = (idx % (K / 4)) * 4;
    const float4 kk = f4(KQ + i * kLd + c), gg = f4(GM + i * kLd + c);
    const float b = bt[i];
    f4(L1 + i * kLd + c) = make_float4(b * kk.x * expf(gg.x), b * kk.y * expf(gg.y),
                                       b * kk.z * expf(gg.z), b * kk.w * expf(gg.w));
  }
  __syncthreads();

  float* rec = a.ws + ((size_t)cid * HV + h) * kRec;
  // 5. W = Ti (beta Ktil): thread owns column quad c4 = lane, rows warp + 8m.
  auto tri_gemm_store = [&](float* dst) {
    const int c = lane * 4;
    for (int t = warp; t < kChunk; t += 8) {
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int i = 0; i <= t; ++i) {
        const float w = Ti[t * kLdT + i];
        const float4 x = f4(L1 + i * kLd + c);
        acc.x += w * x.x;
        acc.y += w * x.y;
        acc.z += w * x.z;
        acc.w += w * x.w;
      }
      f4(dst + t * K + c) = acc;
    }
  };
  tri_gemm_store(rec + kOffW);
  __syncthreads();
  // 6. Util = Ti (beta V)
  for (int idx = tid; idx < kChunk * (K / 4); idx += blockDim.x) {
    const int i = idx / (K / 4), c = (idx % (K / 4)) * 4;
    float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (i < len) vv = load_bf16x4(a.v + ((t0 + i) * HV + h) * K + c);
    const float b = bt[i];
    f4(L1 + i * kLd + c) = make_float4(b * vv.x, b * vv.y, b * vv.z, b * vv.w);
  }
  __syncthreads();
  tri_gemm_store(rec + kOffU);

  // 7. Qtil, Khat, gamma, P
  for (int idx = tid; idx < kChunk * (K / 4); idx += blockDim.x) {
    const int t = idx / (K / 4), c = (idx % (K / 4)) * 4;
    const float4 gg = f4(GM + t * kLd + c), gl = f4(GM + (kChunk - 1) * kLd + c);
    const float4 qq = f4(QQ + t * kLd + c), kk = f4(KQ + t * kLd + c);
    f4(rec + kOffQ + t * K + c) =
        make_float4(qq.x * expf(gg.x), qq.y * expf(gg.y), qq.z * expf(gg.z), qq.w * expf(gg.w));
    f4(rec + kOffKh + t * K + c) =
        make_float4(kk.x * expf(gl.x - gg.x), kk.y * expf(gl.y - gg.y), kk.z * expf(gl.z - gg.z),
                    kk.w * expf(gl.w - gg.w));
  }
  for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x)
    rec[kOffP + idx] = Pm[(idx / kChunk) * kLdT + idx % kChunk];
  if (tid < K) rec[kOffGam + tid] = expf(GM[(kChunk - 1) * kLd + tid]);
}

constexpr size_t kTransformSmem =
    sizeof(float) * (5 * kChunk * kLd + 16 * kLd + 2 * kChunk * kLdT + kChunk);

// ---------------------------------------------------------------------------
// Sequential state pass over the chunks of one sequence, 16 value columns.

constexpr int kVs = 16;      // value columns per CTA
constexpr int kLdS = kVs + 1;

__global__ void __launch_bounds__(256) state_pass_kernel(const PrefillArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* Wm = sm;                   // [64][kLd]
  float* Qm = Wm + kChunk * kLd;    // [64][kLd]
  float* Km = Qm + kChunk * kLd;    // [64][kLd]
  float* Pm = Km + kChunk * kLd;    // [64][kLdT]
  float* Sm = Pm + kChunk * kLdT;   // [128][kLdS]
  float* Um = Sm + kHeadDim * kLdS; // [64][kLdS]
  float* Ut = Um + kChunk * kLdS;   // [64][kLdS]
  float* gm = Ut + kChunk * kLdS;   // [128]
  __shared__ int64_t s_t0, s_t1, s_cbase;
  __shared__ int s_state;

  const int tid = threadIdx.x;
  const int n = blockIdx.z, h = blockIdx.y, v0 = blockIdx.x * kVs;
  const int HV = a.HV, K = kHeadDim, V = kHeadDim;
  if (tid == 0) {
    s_state = 0;
    if (!seqlens_valid(a)) {
      s_state = 2;
      if (blockIdx.x == 0 && h == 0 && n == 0) set_error(a.err_flag, KDA_DEVERR_SEQLENS);
    } else {
      const int slot = a.state_idx[n];
      if (slot < -1 || slot >= a.pool_slots) {
        s_state = 2;
        if (blockIdx.x == 0 && h == 0) set_error(a.err_flag, KDA_DEVERR_SLOT);
      } else if (slot == -1) {
        s_state = 1;
      }
      int64_t base = 0;
      for (int m = 0; m < n; ++m)
        base += (seq_begin(a, m + 1) - seq_begin(a, m) + kChunk - 1) / kChunk;
      s_cbase = base;
      s_t0 = seq_begin(a, n);
      s_t1 = seq_begin(a, n + 1);
    }
  }
  __syncthreads();
  if (s_state == 2) return;
  const int64_t t0 = s_t0, t1 = s_t1;
  if (s_state == 1) {  // padding sequence: zero outputs
    for (int64_t idx = tid; idx < (t1 - t0) * kVs; idx += blockDim.x)
      a.o[((t0 + idx / kVs) * HV + h) * V + v0 + idx % kVs] = 0;
    return;
  }
  const int slot = a.state_idx[n];
  float* st = a.pool + ((size_t)slot * HV + h) * V * K;
  for (int idx = tid; idx < kVs * K; idx += blockDim.x) {
    const int j = idx / K, c = idx % K;
    Sm[c * kLdS + j] = st[(size_t)(v0 + j) * K + c];
  }
  __syncthreads();

  const int nch = (int)((t1 - t0 + kChunk - 1) / kChunk);
  for (int ci = 0; ci < nch; ++ci) {
    const int64_t cid = s_cbase + ci;
    const int64_t tc = t0 + (int64_t)ci * kChunk;
    const int len = (int)(t1 - tc < kChunk ? t1 - tc : kChunk);
    const float* rec = a.ws + ((size_t)cid * HV + h) * kRec;
    if (a.intermediate) {
      float* dst = a.intermediate + ((size_t)cid * HV + h) * V * K;
      for (int idx = tid; idx < kVs * K; idx += blockDim.x) {
        const int j = idx / K, c = idx % K;
        dst[(size_t)(v0 + j) * K + c] = Sm[c * kLdS + j];
      }
    }
    for (int idx = tid; idx < kChunk * (K / 4); idx += blockDim.x) {
      const int t = idx / (K / 4), c = (idx % (K / 4)) * 4;
      f4(Wm + t * kLd + c) = *reinterpret_cast<const float4*>(rec + kOffW + t * K + c);
      f4(Qm + t * kLd + c) = *reinterpret_cast<const float4*>(rec + kOffQ + t * K + c);
      f4(Km + t * kLd + c) = *reinterpret_cast<const float4*>(rec + kOffKh + t * K + c);
    }
    for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x)
      Pm[(idx / kChunk) * kLdT + idx % kChunk] = rec[kOffP + idx];
    for (int idx = tid; idx < kChunk * kVs; idx += blockDim.x)
      Ut[(idx / kVs) * kLdS + idx % kVs] = rec[kOffU + (idx / kVs) * K + v0 + idx % kVs];
    if (tid < K) gm[tid] = rec[kOffGam + tid];
    __syncthreads();

    // U = Util - W S : thread -> (t, 4 columns)
    {
      const int t = tid >> 2, j0 = (tid & 3) * 4;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = 0; c < K; ++c) {
        const float w = Wm[t * kLd + c];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[jj] += w * Sm[c * kLdS + j0 + jj];
      }
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) Um[t * kLdS + j0 + jj] = Ut[t * kLdS + j0 + jj] - acc[jj];
    }
    __syncthreads();
    // O = scale (Qtil S + P U)
    {
      const int t = tid >> 2, j0 = (tid & 3) * 4;
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int c = 0; c < K; ++c) {
        const float w = Qm[t * kLd + c];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[jj] += w * Sm[c * kLdS + j0 + jj];
      }
      for (int i = 0; i <= t; ++i) {
        const float p = Pm[t * kLdT + i];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) acc[jj] += p * Um[i * kLdS + j0 + jj];
      }
      if (t < len) {
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
          a.o[((tc + t) * HV + h) * V + v0 + j0 + jj] = float_to_bf16_bits(a.gate.scale * acc[jj]);
      }
    }
    // S = Diag(gamma) S + Khat^T U : thread -> (c, 8 columns)
    float snew[8];
    {
      const int c = tid >> 1, j0 = (tid & 1) * 8;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) snew[jj] = gm[c] * Sm[c * kLdS + j0 + jj];
      for (int i = 0; i < kChunk; ++i) {
        const float kh = Km[i * kLd + c];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) snew[jj] += kh * Um[i * kLdS + j0 + jj];
      }
    }
    __syncthreads();
    {
      const int c = tid >> 1, j0 = (tid & 1) * 8;
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) Sm[c * kLdS + j0 + jj] = snew[jj];
    }
    __syncthreads();
  }
  for (int idx = tid; idx < kVs * K; idx += blockDim.x) {
    const int j = idx / K, c = idx % K;
    st[(size_t)(v0 + j) * K + c] = Sm[c * kLdS + j];
  }
}

constexpr size_t kPassSmem = sizeof(float) * (3 * kChunk * kLd + kChunk * kLdT + kHeadDim * kLdS +
                                              2 * kChunk * kLdS + kHeadDim);

int64_t max_chunks(int num_seqs, int64_t total_tokens) {
  return total_tokens / kChunk + num_seqs;
}

cudaEvent_t g_stage_events[3] = {nullptr, nullptr, nullptr};

void record_stage(int i, cudaStream_t st) {
  if (g_stage_events[i]) cudaEventRecord(g_stage_events[i], st);
}

}  // namespace
}  // namespace kda

using namespace kda;

extern "C" size_t kda_prefill_workspace_size(kda_dims dims, int num_seqs, int64_t total_tokens) {
  if (num_seqs < 0 || total_tokens < 0 || dims.HV <= 0) return 0;
  return (size_t)max_chunks(num_seqs, total_tokens) * dims.HV * kRec * sizeof(float);
}

extern "C" kda_status kda_prefill(kda_dims dims, kda_gate gate, const kda_bf16* q,
                                  const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                                  const kda_bf16* beta, int64_t gb_rows, float* state_pool,
                                  int pool_slots, const int32_t* state_idx,
                                  const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                                  kda_bf16* o, float* intermediate, void* workspace,
                                  size_t workspace_bytes, int32_t* err_flag, void* stream) {
  kda_status s = check_dims(dims);
  if (s != KDA_OK) return s;
  if (!state_pool || !state_idx) return KDA_ERR_NULL_ARG;  // indexed pool required
  if (num_seqs < 1 || total_tokens < 0 || pool_slots < 0) return KDA_ERR_SHAPE;
  if (gb_rows < total_tokens) return KDA_ERR_SHAPE;  // g/beta must cover every q token
  if (!cu_seqlens && total_tokens % num_seqs != 0) return KDA_ERR_SHAPE;
  if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_NULL_ARG;
  PrefillArgs args{};
  s = check_gate(gate, &args.gate);
  if (s != KDA_OK) return s;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(state_pool) ||
      (intermediate && !aligned16(intermediate)))
    return KDA_ERR_ALIGNMENT;
  const size_t need = kda_prefill_workspace_size(dims, num_seqs, total_tokens);
  if (need > 0 && (!workspace || workspace_bytes < need)) return KDA_ERR_WORKSPACE;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return KDA_ERR_ALIGNMENT;
  args.H = dims.H;
  args.HV = dims.HV;
  args.q = q;
  args.k = k;
  args.v = v;
  args.g = g;
  args.beta = beta;
  args.pool = state_pool;
  args.pool_slots = pool_slots;
  args.state_idx = state_idx;
  args.cu_seqlens = cu_seqlens;
  args.num_seqs = num_seqs;
  args.total_tokens = total_tokens;
  args.o = o;
  args.intermediate = intermediate;
  args.ws = static_cast<float*>(workspace);
  args.err_flag = err_flag;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // Per device and cheap; not a stream operation, so also fine under capture.
  cudaFuncSetAttribute(chunk_transform_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)kTransformSmem);
  cudaFuncSetAttribute(state_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                       (int)kPassSmem);
  const int64_t chunks = max_chunks(num_seqs, total_tokens);
  record_stage(0, st);
  if (chunks > 0) {
    chunk_transform_kernel<<<dim3((unsigned)chunks, dims.HV), 256, kTransformSmem, st>>>(args);
    if ((s = launch_status()) != KDA_OK) return s;
  }
  record_stage(1, st);
  state_pass_kernel<<<dim3(kHeadDim / kVs, dims.HV, num_seqs), 256, kPassSmem, st>>>(args);
  s = launch_status();
  record_stage(2, st);
  return s;
}

extern "C" void kda_prefill_set_stage_events(void* const* events) {
  for (int i = 0; i < 3; ++i)
    g_stage_events[i] = events ? static_cast<cudaEvent_t>(events[i]) : nullptr;
}

extern "C" const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "ok";
    case KDA_ERR_NULL_ARG: return "a required pointer is NULL";
    case KDA_ERR_SHAPE: return "inconsistent shape";
    case KDA_ERR_UNSUPPORTED: return "unsupported shape or option";
    case KDA_ERR_WORKSPACE: return "workspace missing or too small";
    case KDA_ERR_CUDA: return "CUDA launch failed";
    case KDA_ERR_ALIGNMENT: return "pointer or stride not 16-byte aligned";
  }
  return "unknown status";
}
