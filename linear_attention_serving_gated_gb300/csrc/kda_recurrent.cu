// kda_recurrent.cu -- packed decode, chain/tree speculative verify and commit.
//
// Phases (pages): packed single-token decode with the bounded gate routed to
// the packed kernel, and chain/tree target verification that writes a
// per-candidate state snapshot after every draft token ("[KDA] Support Helion
// MTP verification and harden prefill, decode", sglang PR #42857,
// Motivation and Modifications); the decode input contract of
// validate_packed_decode_inputs ("PR #35197 report: fix(kernel) Fix Helion
// small-token prefill bug", kda_decode.py snippet); commit of an accepted
// prefix between verify rounds (PR #42857 review thread).
//
// Design (GB300): these phases move each 64 KiB FP32 head state once per call
// and do ~6 flops per state element per token, so they are HBM-bound.  Every
// thread keeps its share of the state in registers for the whole call:
//   * one CTA = 4 warps covers 16*GROUPS rows j of S^T ([V][K], K contiguous);
//   * a warp works on 4 rows at once, 8 lanes per row, each lane holding 16
//     key channels c = i*32 + sub*4 + {0..3} (i < 4) as four float4, so each
//     128-bit load instruction reads four full 128-byte row segments;
//   * k^T x and S^T q are 16-term packed-FP32 (f32x2) partial dots finished
//     with three xor-shuffles inside the 8-lane row group;
//   * the fold (L2 norm, gate, sigmoid beta) of up to 8 tokens at a time is
//     computed once per CTA, one key channel per thread, into shared memory;
//     lanes then read their 16 channels as float4 (broadcast across the
//     four row groups of a warp);
//   * verify keeps the state in registers across the T draft tokens and
//     writes each snapshot straight from registers; a tree node whose parent
//     is not the previous node reloads the parent's snapshot, which this same
//     thread wrote (so it is visible to it without any barrier); snapshots
//     that will be reloaded are stored with L1 evict-last priority, the
//     others without allocating in L1.
#include <atomic>

#include "kda_host.h"

namespace kda {
namespace {

// kChainReplay: chain verify that keeps no snapshots; instead each draft
// token's folded inputs go to a per-request ring.  kCommitReplay: replays the
// accepted prefix from that ring onto the pool state.  kSeqPrefill: a
// prefill's sequences token by token (o, chunk-start states, final state),
// for log-decays the chunk form's decay windows cannot take.
enum Mode { kDecode = 0, kChain = 1, kTree = 2, kChainReplay = 3, kCommitReplay = 4, kSeqPrefill = 5 };
constexpr int kSeqChunk = 64;  // the prefill's chunk length (chunk-start states)

// Ring record of one (request, token, head): k-hat [128], exp(g) [128],
// v [128], beta, padding -- FP32, 16-byte aligned.
constexpr int kRingFloats = 3 * kHeadDim + 4;

struct StepArgs {
  GateArgs gate;
  int H, HV;
  int G;      // value heads per q/k head (HV / H)
  int dtype;  // KDA_DTYPE_BF16 or KDA_DTYPE_F16: token rows and o
  const kda_bf16* mixed_qkv;
  int64_t row_stride;
  const kda_bf16* a;
  const kda_bf16* b;
  int B, T;
  const int32_t* parent;
  float* pool;
  int pool_slots;
  const int32_t* state_idx;
  kda_bf16* o;
  float* snapshots;
  float* ring;                // replay modes
  const int32_t* accepted;    // kCommitReplay
  int32_t* err_flag;
  // kSeqPrefill: q, k [T][H][K] and v [T][HV][V] (the gate input is a, beta
  // is b), sequence bounds, which sequences run, chunk-start states
  const kda_bf16 *sq, *sk, *sv;
  const int32_t* cu_seqlens;
  int num_seqs;
  int64_t total_tokens;
  const int32_t* seq_flags;  // non-null: only flagged sequences run
  float* intermediate;
  int64_t inter_chunks;
  const int64_t* chunk_base;  // [num_seqs] chunk id of each sequence's first chunk
  int seq0;                   // sequence of blockIdx.z == 0 (launches of at most 65535)
};

__device__ __forceinline__ int64_t seq_start(const StepArgs& a, int n) {
  return a.cu_seqlens ? (int64_t)a.cu_seqlens[n] : a.total_tokens / a.num_seqs * n;
}

__device__ __forceinline__ float group_sum8(float x) {
  x += __shfl_xor_sync(0xffffffffu, x, 1);
  x += __shfl_xor_sync(0xffffffffu, x, 2);
  x += __shfl_xor_sync(0xffffffffu, x, 4);
  return x;
}

// Tree verify's snapshot stores: a snapshot that a later node reloads (its
// parent is not the node just before it) stays in L1 with evict-last
// priority, so that the reload, by the same thread, finds it there; the
// others are not allocated in L1, which keeps room for the kept ones.
__device__ __forceinline__ void st_keep_l1(float* p, float4 v) {
  asm volatile("st.global.L1::evict_last.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}
__device__ __forceinline__ void st_skip_l1(float* p, float4 v) {
  asm volatile("st.global.L1::no_allocate.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}
// The state of decode and ReplaySSM verify (CTAs of two or more row groups)
// is read once and, for decode, written once: neither needs L1.
__device__ __forceinline__ float4 ld_skip_l1(const float* p) {
  float4 v;
  asm volatile("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float dot16(const float4 (&x)[4], const float4 (&y)[4]) {
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc = fma2(make_float2(x[i].x, x[i].y), make_float2(y[i].x, y[i].y), acc);
    acc = fma2(make_float2(x[i].z, x[i].w), make_float2(y[i].z, y[i].w), acc);
  }
  return acc.x + acc.y;
}

constexpr int kTokBlock = 8;  // tokens folded per shared-memory pass

struct FoldSmem {
  float q[kTokBlock][kHeadDim];    // q-hat
  float k[kTokBlock][kHeadDim];    // k-hat
  float dec[kTokBlock][kHeadDim];  // exp(g)
  float v[kTokBlock][kHeadDim];
  float gbias[kHeadDim];           // ReplaySSM verify: dt_bias of the head, and
  float galog;                     // A_log, copied with the token rows
  float beta[kTokBlock];
  float red[kTokBlock][2][4];      // per-warp sums of squares of q and k
};

// CTAs per SM the register allocation must allow: 7 (72 registers) lets the
// 1024 CTAs of a 16-request verify run as one wave (tree verify fits there
// with its row groups stepped together).  Four row groups (64-row CTAs of
// tree and ReplaySSM verify, up to 128 registers) run 4 per SM, and so does
// the prefill's token-by-token path, which would spill at 72.
template <int MODE, int GROUPS>
constexpr int kMinCtasPerSm = GROUPS == 4 || MODE == kSeqPrefill ? 4 : 7;

template <int MODE, int GROUPS, bool F16>
__global__ void __launch_bounds__(128, (kMinCtasPerSm<MODE, GROUPS>)) recurrent_kernel(const StepArgs args) {
  constexpr int K = kHeadDim, V = kHeadDim;
  __shared__ __align__(16) FoldSmem fs;
  __shared__ int tree_par[kTokBlock];  // tree: the parents of the first kTokBlock nodes
  __shared__ uint32_t tree_keep;       // tree: bit i, node i's snapshot is reloaded by a later node
  // raw BF16 token rows of this head: q, k, v, gate input, per token of the block
  __shared__ __align__(16) uint16_t raw_s[kTokBlock][4][kHeadDim];
  const int r = blockIdx.z + (MODE == kSeqPrefill ? args.seq0 : 0), h = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int sub = lane & 7;
  const int row0 = blockIdx.x * (16 * GROUPS) + warp * (4 * GROUPS) + (lane >> 3);
  const int HV = args.HV;
  const bool reporter = tid == 0 && blockIdx.x == 0 && h == 0;
  // commit replay: the ring records of the first block are copied into the
  // fold buffers before the accepted index is known (4-byte and 16-byte
  // asynchronous copies), then tokens 0..accepted[r] are replayed
  if (MODE == kCommitReplay) {
    const int n0 = args.T < kTokBlock ? args.T : kTokBlock;
    for (int idx = tid; idx < n0 * 3 * 32; idx += 128) {
      const int u = idx / 96, part = idx % 96, m = part >> 5, piece = (part & 31) * 4;
      const float* rec = args.ring + (((int64_t)r * args.T + u) * args.HV + h) * kRingFloats;
      float* dst = m == 0 ? &fs.k[u][piece] : m == 1 ? &fs.dec[u][piece] : &fs.v[u][piece];
      cp_async16(dst, rec + m * kHeadDim + piece);
    }
    if (tid < n0)
      cp_async4(&fs.beta[tid], args.ring + (((int64_t)r * args.T + tid) * args.HV + h) * kRingFloats +
                                   3 * kHeadDim);
    cp_async_commit();
  }
  const int acc = MODE == kCommitReplay ? args.accepted[r] : 0;
  if (MODE == kCommitReplay) {
    if (acc < 0 || acc >= args.T) {
      if (acc >= args.T && reporter) set_error(args.err_flag, KDA_DEVERR_ACCEPTED);
      cp_async_wait_all();  // no copy into shared memory outlives the CTA
      return;  // acc < 0: nothing accepted, the pool keeps its state
    }
  }
  // kSeqPrefill: request r is sequence r, its tokens [sp_t0, sp_t0 + T)
  int64_t sp_t0 = 0, sp_cbase = 0;
  int sp_T = 0;
  if constexpr (MODE == kSeqPrefill) {
    if (args.seq_flags && !args.seq_flags[r]) return;  // this sequence took the chunk form
    sp_t0 = seq_start(args, r);
    const int64_t sp_t1 = seq_start(args, r + 1);
    if (sp_t0 < 0 || sp_t1 < sp_t0 || sp_t1 > args.total_tokens) {  // no access outside the token rows
      if (reporter) set_error(args.err_flag, KDA_DEVERR_SEQLENS);
      return;
    }
    sp_T = (int)(sp_t1 - sp_t0);
    if (sp_T == 0) return;  // keeps its state
    if (args.intermediate) sp_cbase = args.chunk_base[r];
  }
  const int T = MODE == kDecode ? 1 : MODE == kCommitReplay ? acc + 1 : MODE == kSeqPrefill ? sp_T : args.T;
  // the o row of token t
  auto out_row = [&](int t) -> int64_t {
    return MODE == kDecode ? r : MODE == kSeqPrefill ? sp_t0 + t : (int64_t)r * T + t;
  };

  // Raw token rows of a block, copied 16 bytes at a time into raw_s.  The
  // first block's copies are issued before anything that waits on memory,
  // so their latency overlaps the slot lookup and the state load.
  // Thread tid copies 16-byte piece tid % 16 of tensor (tid / 16) % 4 (q, k,
  // v of a packed row, or the gate input row) of tokens tid / 64, +2, ...:
  // its element offset within the row is fixed.  Value head h reads q/k head
  // h / G.
  const int raw_m = (tid >> 4) & 3, raw_piece = (tid & 15) * 8;
  const int raw_off = MODE == kCommitReplay ? 0  // reads no token rows
                    : MODE == kSeqPrefill ? raw_piece + (raw_m < 2 ? h / args.G : h) * kHeadDim  // separate tensors
                    : raw_piece + (raw_m == 0 ? (h / args.G) * kHeadDim
                                 : raw_m == 1 ? (args.H + h / args.G) * kHeadDim
                                 : raw_m == 2 ? (2 * args.H + h) * kHeadDim
                                              : h * kHeadDim);
  uint16_t b_raw = 0;  // thread u < nt: raw beta of token u of the block
  auto request_raw = [&](int tb, int nt) {
    for (int u = tid >> 6; u < nt; u += 2) {
      const int64_t row = out_row(tb + u);
      const kda_bf16* x;
      if constexpr (MODE == kSeqPrefill)
        x = raw_m == 0 ? args.sq + row * ((int64_t)args.H * kHeadDim)
          : raw_m == 1 ? args.sk + row * ((int64_t)args.H * kHeadDim)
          : raw_m == 2 ? args.sv + row * ((int64_t)args.HV * kHeadDim)
                       : args.a + row * ((int64_t)args.HV * kHeadDim);
      else
        x = raw_m < 3 ? args.mixed_qkv + row * args.row_stride : args.a + row * ((int64_t)args.HV * kHeadDim);
      cp_async16(&raw_s[u][raw_m][raw_piece], x + raw_off);
    }
    cp_async_commit();
    if (tid < nt) {  // kept in a register: its latency overlaps the slot lookup and state load
      const int64_t row = out_row(tb + tid);
      b_raw = args.b[row * args.HV + h];
    }
  };
  if (MODE != kCommitReplay) request_raw(0, T < kTokBlock ? T : kTokBlock);
  // Gate parameters: loaded before the slot lookup so that their latency
  // overlaps it.  ReplaySSM verify, where a longer live range spills at its
  // register budget, copies them into shared memory with the token rows
  // instead.  exp(A_log) is taken after the state load.
  constexpr bool kEarlyGate = MODE != kChainReplay;
  const GateArgs& ga = args.gate;
  float alog_early = 0.f, bias_early = 0.f;
  if constexpr (kEarlyGate) {
    alog_early = ga.A_log ? ga.A_log[h] : 0.f;
    bias_early = ga.dt_bias ? ga.dt_bias[h * K + tid] : 0.f;
  } else {
    if (ga.dt_bias && tid < kHeadDim / 4) cp_async16(&fs.gbias[tid * 4], ga.dt_bias + h * K + tid * 4);
    if (ga.A_log && tid == kHeadDim / 4) cp_async4(&fs.galog, ga.A_log + h);
    cp_async_commit();
  }

  const int slot = args.state_idx[r];
  const bool ok = slot >= -1 && slot < args.pool_slots;
  if (!ok && reporter) set_error(args.err_flag, KDA_DEVERR_SLOT);
  // Tree: a request with a parent outside [-1, i) is rejected.  It runs down
  // the chain path (no parent reloads), writes no snapshot and zero outputs,
  // so the rejection adds no branch around the main loop.
  bool parents_ok = true;
  if (MODE == kTree && ok && slot >= 0) {
    bool bad = false;
    for (int i = tid; i < T; i += 128) {
      const int p = args.parent[(int64_t)r * T + i];
      bad |= p < -1 || p >= i;
    }
    if (tid < kTokBlock && tid < T) tree_par[tid] = args.parent[(int64_t)r * T + tid];
    parents_ok = !__syncthreads_or(bad);
    if (tid == 0) {  // read after the fold's barriers; past kTokBlock nodes, every snapshot is kept
      uint32_t keep = T > kTokBlock ? 0xffffffffu : 0u;
      for (int i = 1; i < T && i < kTokBlock; ++i) {
        const int p = tree_par[i];
        if (p >= 0 && p != i - 1) keep |= 1u << p;
      }
      tree_keep = keep;
    }
    if (!parents_ok && reporter) set_error(args.err_flag, KDA_DEVERR_PARENT);
  }
  if (!ok || slot < 0) {  // padding or rejected request: zero outputs, touch no state
    cp_async_wait_all();  // no copy into shared memory outlives the CTA
    if (MODE != kCommitReplay && sub == 0)
      for (int i = 0; i < T; ++i)
#pragma unroll
        for (int gi = 0; gi < GROUPS; ++gi)
          args.o[(out_row(i) * HV + h) * V + row0 + gi * 4] = 0;
    return;
  }

  const size_t head_elems = (size_t)V * K;
  float* root = args.pool + ((size_t)slot * HV + h) * head_elems;
  const int lane_col = sub * 4;

  float4 S[GROUPS][4];
#pragma unroll
  for (int gi = 0; gi < GROUPS; ++gi)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      S[gi][i] = (MODE == kDecode || MODE == kChainReplay) && GROUPS >= 2
                     ? ld_skip_l1(root + (size_t)(row0 + gi * 4) * K + i * 32 + lane_col)
                     : *reinterpret_cast<const float4*>(root + (size_t)(row0 + gi * 4) * K + i * 32 + lane_col);

  // (ReplaySSM verify: set once its copies have landed, in the first fold)
  float exp_alog = kEarlyGate && ga.A_log ? __expf(alog_early) : 0.f;
  float bias_c = kEarlyGate ? bias_early : 0.f;

  for (int tb = 0; tb < T; tb += kTokBlock) {
    const int nt = T - tb < kTokBlock ? T - tb : kTokBlock;
    // fold of tokens [tb, tb+nt): thread tid owns key channel / value column tid
    if (MODE != kCommitReplay && tb > 0) request_raw(tb, nt);
    if (tb == 0 || MODE != kCommitReplay) {
      cp_async_wait_all();
      __syncthreads();
    }
    if (!kEarlyGate && tb == 0) {
      exp_alog = ga.A_log ? __expf(fs.galog) : 0.f;
      bias_c = ga.dt_bias ? fs.gbias[tid] : 0.f;
    }
    float sq[kTokBlock], sk[kTokBlock];
#pragma unroll
    for (int u = 0; u < kTokBlock; ++u) {
      sq[u] = 0.f;
      sk[u] = 0.f;
      if (MODE == kCommitReplay) {  // folded values recorded by the verify
        if (u < nt && tb > 0) {  // the first block arrived by asynchronous copies
          const float* rec = args.ring + (((int64_t)r * args.T + tb + u) * HV + h) * kRingFloats;
          fs.k[u][tid] = rec[tid];
          fs.dec[u][tid] = rec[kHeadDim + tid];
          fs.v[u][tid] = rec[2 * kHeadDim + tid];
          if (tid == 0) fs.beta[u] = rec[3 * kHeadDim];
        }
      } else if (u < nt) {
        const float qv = in16_to_float<F16>(raw_s[u][0][tid]);
        const float kv = in16_to_float<F16>(raw_s[u][1][tid]);
        const float av = in16_to_float<F16>(raw_s[u][3][tid]);
        fs.q[u][tid] = qv;
        fs.k[u][tid] = kv;
        fs.v[u][tid] = in16_to_float<F16>(raw_s[u][2][tid]);
        fs.dec[u][tid] = decay_exp(gate_log_decay(ga, av, exp_alog, bias_c));
        sq[u] = qv * qv;
        sk[u] = kv * kv;
      }
    }
    if (MODE != kCommitReplay && tid < nt) fs.beta[tid] = fold_beta(ga, in16_to_float<F16>(b_raw));
    if (MODE != kCommitReplay && ga.use_qk_l2norm) {
#pragma unroll
      for (int u = 0; u < kTokBlock; ++u) {
        if (u < nt) {  // nt is the same in every thread
#pragma unroll
          for (int m = 16; m; m >>= 1) {
            sq[u] += __shfl_xor_sync(0xffffffffu, sq[u], m);
            sk[u] += __shfl_xor_sync(0xffffffffu, sk[u], m);
          }
          if (lane == 0) {
            fs.red[u][0][warp] = sq[u];
            fs.red[u][1][warp] = sk[u];
          }
        }
      }
      __syncthreads();
#pragma unroll
      for (int u = 0; u < kTokBlock; ++u) {
        if (u < nt) {
          const float rq = rsqrtf(fs.red[u][0][0] + fs.red[u][0][1] + fs.red[u][0][2] +
                                  fs.red[u][0][3] + kNormEps);
          const float rk = rsqrtf(fs.red[u][1][0] + fs.red[u][1][1] + fs.red[u][1][2] +
                                  fs.red[u][1][3] + kNormEps);
          fs.q[u][tid] *= rq;
          fs.k[u][tid] *= rk;
        }
      }
    }
    __syncthreads();
    for (int u = 0; u < nt; ++u) {
      const int t = tb + u;
      if (MODE == kChainReplay && blockIdx.x == 0) {  // one row block per head records the fold
        float* rec = args.ring + (((int64_t)r * T + t) * HV + h) * kRingFloats;
        rec[tid] = fs.k[u][tid];
        rec[kHeadDim + tid] = fs.dec[u][tid];
        rec[2 * kHeadDim + tid] = fs.v[u][tid];
        if (tid == 0) rec[3 * kHeadDim] = fs.beta[u];
      }
      if (MODE == kTree && t > 0 && parents_ok) {
        const int p = t < kTokBlock ? tree_par[t] : args.parent[(int64_t)r * T + t];
        if (p != t - 1) {
          const float* src =
              p < 0 ? root : args.snapshots + (((size_t)r * T + p) * HV + h) * head_elems;
#pragma unroll
          for (int gi = 0; gi < GROUPS; ++gi)
#pragma unroll
            for (int i = 0; i < 4; ++i)
              S[gi][i] = *reinterpret_cast<const float4*>(src + (size_t)(row0 + gi * 4) * K +
                                                          i * 32 + lane_col);
        }
      }
      const int64_t row = out_row(t);
      if constexpr (MODE == kSeqPrefill) {  // the state at the start of each chunk
        if (args.intermediate && t % kSeqChunk == 0) {
          const int64_t cid = sp_cbase + t / kSeqChunk;
          if (cid >= 0 && cid < args.inter_chunks) {
            float* dst = args.intermediate + (size_t)(cid * HV + h) * head_elems;
#pragma unroll
            for (int gi = 0; gi < GROUPS; ++gi)
#pragma unroll
              for (int i = 0; i < 4; ++i)
                *reinterpret_cast<float4*>(dst + (size_t)(row0 + gi * 4) * K + i * 32 + lane_col) = S[gi][i];
          } else if (reporter) {
            set_error(args.err_flag, KDA_DEVERR_INTERMEDIATE);
          }
        }
      }
      float4 q[4], k[4], dec[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        q[i] = *reinterpret_cast<const float4*>(&fs.q[u][i * 32 + lane_col]);
        k[i] = *reinterpret_cast<const float4*>(&fs.k[u][i * 32 + lane_col]);
        dec[i] = *reinterpret_cast<const float4*>(&fs.dec[u][i * 32 + lane_col]);
      }
      const float beta = fs.beta[u];
      float* snap = MODE == kChain || MODE == kTree
                        ? args.snapshots + (((size_t)r * T + t) * HV + h) * head_elems
                        : nullptr;
      if constexpr (MODE == kTree) {
        // X = Diag(exp g) S;  u = beta (v - X^T k);  S = X + k u^T;  o = scale S^T q.
        // The row groups go through each step together, so that one group's
        // dot, shuffle and update latencies overlap the others'.
        float pk[GROUPS], po[GROUPS];
#pragma unroll
        for (int gi = 0; gi < GROUPS; ++gi) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 lo = mul2(make_float2(S[gi][i].x, S[gi][i].y), make_float2(dec[i].x, dec[i].y));
            const float2 hi = mul2(make_float2(S[gi][i].z, S[gi][i].w), make_float2(dec[i].z, dec[i].w));
            S[gi][i] = make_float4(lo.x, lo.y, hi.x, hi.y);
          }
          pk[gi] = dot16(S[gi], k);
        }
#pragma unroll
        for (int m = 1; m < 8; m <<= 1)  // the 8-lane row group's sums, as group_sum8
#pragma unroll
          for (int gi = 0; gi < GROUPS; ++gi) pk[gi] += __shfl_xor_sync(0xffffffffu, pk[gi], m);
#pragma unroll
        for (int gi = 0; gi < GROUPS; ++gi) {
          const float uu = beta * (fs.v[u][row0 + gi * 4] - pk[gi]);
          const float2 u2 = make_float2(uu, uu);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 lo = fma2(make_float2(k[i].x, k[i].y), u2, make_float2(S[gi][i].x, S[gi][i].y));
            const float2 hi = fma2(make_float2(k[i].z, k[i].w), u2, make_float2(S[gi][i].z, S[gi][i].w));
            S[gi][i] = make_float4(lo.x, lo.y, hi.x, hi.y);
          }
          if (MODE != kCommitReplay) po[gi] = dot16(S[gi], q);
        }
        if (MODE == kCommitReplay) continue;  // the state is written once, after the last token
#pragma unroll
        for (int m = 1; m < 8; m <<= 1)
#pragma unroll
          for (int gi = 0; gi < GROUPS; ++gi) po[gi] += __shfl_xor_sync(0xffffffffu, po[gi], m);
#pragma unroll
        for (int gi = 0; gi < GROUPS; ++gi) {
          const int j = row0 + gi * 4;
          const float out = ga.scale * po[gi];
          if (sub == 0) args.o[(row * HV + h) * V + j] = parents_ok ? float_to_out16<F16>(out) : 0;
          if (MODE != kChainReplay && (MODE != kTree || parents_ok)) {  // ReplaySSM verify keeps no snapshots
            float* dst = MODE == kDecode ? root + (size_t)j * K : snap + (size_t)j * K;
            if (t >= 32 || (tree_keep >> t & 1u)) {
#pragma unroll
              for (int i = 0; i < 4; ++i) st_keep_l1(dst + i * 32 + lane_col, S[gi][i]);
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) st_skip_l1(dst + i * 32 + lane_col, S[gi][i]);
            }
          }
        }
      } else {
#pragma unroll
        for (int gi = 0; gi < GROUPS; ++gi) {
          // X = Diag(exp g) S;  u = beta (v - X^T k);  S = X + k u^T;  o = scale S^T q
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 lo = mul2(make_float2(S[gi][i].x, S[gi][i].y), make_float2(dec[i].x, dec[i].y));
            const float2 hi = mul2(make_float2(S[gi][i].z, S[gi][i].w), make_float2(dec[i].z, dec[i].w));
            S[gi][i] = make_float4(lo.x, lo.y, hi.x, hi.y);
          }
          const int j = row0 + gi * 4;
          const float uu = beta * (fs.v[u][j] - group_sum8(dot16(S[gi], k)));
          const float2 u2 = make_float2(uu, uu);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 lo = fma2(make_float2(k[i].x, k[i].y), u2, make_float2(S[gi][i].x, S[gi][i].y));
            const float2 hi = fma2(make_float2(k[i].z, k[i].w), u2, make_float2(S[gi][i].z, S[gi][i].w));
            S[gi][i] = make_float4(lo.x, lo.y, hi.x, hi.y);
          }
          if (MODE == kCommitReplay) continue;  // the state is written once, after the last token
          const float out = ga.scale * group_sum8(dot16(S[gi], q));
          if (sub == 0) args.o[(row * HV + h) * V + j] = parents_ok ? float_to_out16<F16>(out) : 0;
          if (MODE == kChainReplay || MODE == kSeqPrefill) continue;  // no snapshots
          if (MODE != kTree || parents_ok) {
            float* dst = MODE == kDecode ? root + (size_t)j * K : snap + (size_t)j * K;
            if (MODE == kDecode && GROUPS >= 2) {
#pragma unroll
              for (int i = 0; i < 4; ++i) st_skip_l1(dst + i * 32 + lane_col, S[gi][i]);
            } else {
#pragma unroll
              for (int i = 0; i < 4; ++i) *reinterpret_cast<float4*>(dst + i * 32 + lane_col) = S[gi][i];
            }
          }
        }
      }
    }
    if (tb + kTokBlock < T) __syncthreads();  // fold buffer reused by the next block
  }
  if (MODE == kCommitReplay || MODE == kSeqPrefill) {  // the final state, once
#pragma unroll
    for (int gi = 0; gi < GROUPS; ++gi)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<float4*>(root + (size_t)(row0 + gi * 4) * K + i * 32 + lane_col) = S[gi][i];
  }
}

constexpr int kCommitVec = 4;  // float4 per thread

__global__ void __launch_bounds__(256) commit_kernel(const float* __restrict__ snapshots, int T,
                                                     const int32_t* __restrict__ accepted,
                                                     float* __restrict__ pool, int pool_slots,
                                                     const int32_t* __restrict__ state_idx,
                                                     size_t slot_elems, int32_t* err_flag) {
  const int r = blockIdx.y;
  const int acc = accepted[r];
  const int slot = state_idx[r];
  const bool reporter = threadIdx.x == 0 && blockIdx.x == 0;
  if (acc < 0) return;
  if (acc >= T) {
    if (reporter) set_error(err_flag, KDA_DEVERR_ACCEPTED);
    return;
  }
  if (slot < -1 || slot >= pool_slots) {
    if (reporter) set_error(err_flag, KDA_DEVERR_SLOT);
    return;
  }
  if (slot < 0) return;
  const float4* src = reinterpret_cast<const float4*>(snapshots + ((size_t)r * T + acc) * slot_elems);
  float4* dst = reinterpret_cast<float4*>(pool + (size_t)slot * slot_elems);
  const size_t n4 = slot_elems / 4;
  // each thread moves kCommitVec float4 spaced blockDim.x apart, with all its
  // loads in flight before the first store
  const size_t base = (size_t)blockIdx.x * blockDim.x * kCommitVec + threadIdx.x;
  float4 v[kCommitVec];
#pragma unroll
  for (int e = 0; e < kCommitVec; ++e) {
    const size_t i = base + (size_t)e * blockDim.x;
    if (i < n4) v[e] = __ldcs(src + i);
  }
#pragma unroll
  for (int e = 0; e < kCommitVec; ++e) {
    const size_t i = base + (size_t)e * blockDim.x;
    if (i < n4) dst[i] = v[e];
  }
}

// SMs of the current device (looked up once per device).
int sm_count() {
  static std::atomic<int> counts[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  int n = counts[dev].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    counts[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <int MODE>
kda_status launch_recurrent(const StepArgs& a, cudaStream_t stream, bool stages = true) {
  // Small batches use 16-row CTAs so that even one request spreads over 128
  // CTAs; larger batches use 32-row CTAs to halve the per-CTA fold work.
  // Tree verify takes 64-row CTAs where their grid fits in one wave and the
  // 32-row one does not (at 16 heads, 17 to 19 requests).  ReplaySSM verify,
  // bound by its per-token steps and the fold rather than by bytes, takes
  // them wherever they fill the SMs in one wave (at 16 heads, 5 to 19
  // requests): half as many CTAs fold each request's tokens.
  const int64_t units = (int64_t)a.B * a.HV;
  const int sms = sm_count();
  if (sms <= 0) return KDA_ERR_CUDA;
  if (stages) record_stage(0, stream);
  const bool f16 = a.dtype == KDA_DTYPE_F16;
  if (units * 8 <= 2 * (int64_t)sms) {
    dim3 grid(kHeadDim / 16, a.HV, a.B);
    (f16 ? recurrent_kernel<MODE, 1, true> : recurrent_kernel<MODE, 1, false>)<<<grid, 128, 0, stream>>>(a);
  } else if ((MODE == kTree && units * (kHeadDim / 32) > (int64_t)kMinCtasPerSm<MODE, 2> * sms &&
              units * (kHeadDim / 64) <= (int64_t)kMinCtasPerSm<MODE, 4> * sms) ||
             (MODE == kChainReplay && units * (kHeadDim / 64) >= sms &&
              units * (kHeadDim / 64) <= (int64_t)kMinCtasPerSm<MODE, 4> * sms)) {
    if constexpr (MODE == kTree || MODE == kChainReplay) {
      dim3 grid(kHeadDim / 64, a.HV, a.B);
      (f16 ? recurrent_kernel<MODE, 4, true> : recurrent_kernel<MODE, 4, false>)<<<grid, 128, 0, stream>>>(a);
    }
  } else {
    dim3 grid(kHeadDim / 32, a.HV, a.B);
    (f16 ? recurrent_kernel<MODE, 2, true> : recurrent_kernel<MODE, 2, false>)<<<grid, 128, 0, stream>>>(a);
  }
  const kda_status s = launch_status();
  if (stages) {
    record_stage(1, stream);
    record_stage(2, stream);
  }
  return s;
}

kda_status check_packed(const kda_dims& dims, const kda_gate& gate, const kda_bf16* mixed_qkv,
                        int64_t row_stride, const kda_bf16* a, const kda_bf16* b, int B,
                        const void* pool, int pool_slots, const int32_t* state_idx,
                        const kda_bf16* o, StepArgs* out) {
  kda_status s = check_dims(dims);
  if (s != KDA_OK) return s;
  if (!pool || !state_idx) return KDA_ERR_NULL_ARG;
  if (B < 0 || pool_slots < 0) return KDA_ERR_SHAPE;
  if (B > 0 && (!mixed_qkv || !a || !b || !o)) return KDA_ERR_NULL_ARG;
  if (row_stride < 2 * (int64_t)dims.H * dims.K + (int64_t)dims.HV * dims.V)
    return KDA_ERR_SHAPE;
  if (row_stride % 8 != 0 || !aligned16(mixed_qkv) || !aligned16(a) || !aligned16(pool))
    return KDA_ERR_ALIGNMENT;
  s = check_gate(gate, &out->gate);
  if (s != KDA_OK) return s;
  out->H = dims.H;
  out->HV = dims.HV;
  out->G = dims.HV / dims.H;
  out->dtype = dims.dtype;
  out->mixed_qkv = mixed_qkv;
  out->row_stride = row_stride;
  out->a = a;
  out->b = b;
  out->B = B;
  out->pool_slots = pool_slots;
  out->state_idx = state_idx;
  return KDA_OK;
}

// The chunk id of each sequence's first chunk: the exclusive prefix sum of
// the per-sequence chunk counts, 1024 sequences per round with the running
// total carried.  One CTA; empty or malformed sequences count 0 chunks (the
// token path checks their bounds itself).
__global__ void __launch_bounds__(1024) seq_chunk_base_kernel(const StepArgs a, int64_t* base) {
  __shared__ int64_t warp_total[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int64_t carry = 0;
  for (int n0 = 0; n0 < a.num_seqs; n0 += 1024) {
    const int n = n0 + tid;
    int64_t c = 0;
    if (n < a.num_seqs) {
      const int64_t L = seq_start(a, n + 1) - seq_start(a, n);
      c = L > 0 ? (L + kSeqChunk - 1) / kSeqChunk : 0;
    }
    int64_t x = c;  // inclusive scan within the warp
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    if (lane == 31) warp_total[warp] = x;
    __syncthreads();
    if (warp == 0) {  // inclusive scan of the warp totals
      int64_t w = warp_total[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int64_t y = __shfl_up_sync(0xffffffffu, w, d);
        if (lane >= d) w += y;
      }
      warp_total[lane] = w;
    }
    __syncthreads();
    if (n < a.num_seqs) base[n] = carry + (warp ? warp_total[warp - 1] : 0) + x - c;
    carry += warp_total[31];
    __syncthreads();  // warp_total is rewritten by the next round
  }
}

}  // namespace

// The prefill's token-by-token path (see kSeqPrefill).
kda_status launch_seq_prefill(const SeqPrefillArgs& p, cudaStream_t stream) {
  if (p.num_seqs <= 0 || p.total_tokens <= 0) return KDA_OK;
  StepArgs a{};
  a.gate = p.gate;
  a.H = p.dims.H;
  a.HV = p.dims.HV;
  a.G = p.dims.HV / p.dims.H;
  a.dtype = p.dims.dtype;
  a.sq = p.q;
  a.sk = p.k;
  a.sv = p.v;
  a.a = p.g;
  a.b = p.beta;
  a.B = p.num_seqs;
  a.pool = p.pool;
  a.pool_slots = p.pool_slots;
  a.state_idx = p.state_idx;
  a.o = p.o;
  a.err_flag = p.err_flag;
  a.cu_seqlens = p.cu_seqlens;
  a.num_seqs = p.num_seqs;
  a.total_tokens = p.total_tokens;
  a.seq_flags = p.seq_flags;
  a.intermediate = p.intermediate;
  a.inter_chunks = p.inter_chunks;
  a.chunk_base = p.chunk_base;
  if (p.intermediate) {
    seq_chunk_base_kernel<<<1, 1024, 0, stream>>>(a, p.chunk_base);
    const kda_status s = launch_status();
    if (s != KDA_OK) return s;
  }
  constexpr int kMaxGridZ = 65535;
  for (int s0 = 0; s0 < p.num_seqs; s0 += kMaxGridZ) {
    a.seq0 = s0;
    a.B = p.num_seqs - s0 < kMaxGridZ ? p.num_seqs - s0 : kMaxGridZ;
    const kda_status s = launch_recurrent<kSeqPrefill>(a, stream, false);
    if (s != KDA_OK) return s;
  }
  return KDA_OK;
}
}  // namespace kda

using namespace kda;

extern "C" kda_status kda_decode_packed(kda_dims dims, kda_gate gate, const kda_bf16* mixed_qkv,
                                        int64_t row_stride, const kda_bf16* a, const kda_bf16* b,
                                        int B, float* state_pool, int pool_slots,
                                        const int32_t* state_idx, kda_bf16* o, int32_t* err_flag,
                                        void* stream) {
  StepArgs args{};
  kda_status s = check_packed(dims, gate, mixed_qkv, row_stride, a, b, B, state_pool, pool_slots,
                              state_idx, o, &args);
  if (s != KDA_OK) return s;
  if (B == 0) return KDA_OK;
  args.T = 1;
  args.pool = state_pool;
  args.o = o;
  args.err_flag = err_flag;
  return launch_recurrent<kDecode>(args, static_cast<cudaStream_t>(stream));
}

static kda_status verify_common(kda_dims dims, kda_gate gate, const kda_bf16* mixed_qkv,
                                int64_t row_stride, const kda_bf16* a, const kda_bf16* b, int B,
                                int T, const int32_t* parent_idx, const float* state_pool,
                                int pool_slots, const int32_t* state_idx, kda_bf16* o,
                                float* snapshots, int32_t* err_flag, void* stream, bool tree) {
  StepArgs args{};
  kda_status s = check_packed(dims, gate, mixed_qkv, row_stride, a, b, B, state_pool, pool_slots,
                              state_idx, o, &args);
  if (s != KDA_OK) return s;
  if (T < 1) return KDA_ERR_SHAPE;
  if (B == 0) return KDA_OK;
  if (!snapshots || (tree && !parent_idx)) return KDA_ERR_NULL_ARG;
  if (!aligned16(snapshots)) return KDA_ERR_ALIGNMENT;
  args.T = T;
  args.parent = parent_idx;
  args.pool = const_cast<float*>(state_pool);  // read only in verify
  args.o = o;
  args.snapshots = snapshots;
  args.err_flag = err_flag;
  return tree ? launch_recurrent<kTree>(args, static_cast<cudaStream_t>(stream))
              : launch_recurrent<kChain>(args, static_cast<cudaStream_t>(stream));
}

extern "C" kda_status kda_verify_chain(kda_dims dims, kda_gate gate, const kda_bf16* mixed_qkv,
                                       int64_t row_stride, const kda_bf16* a, const kda_bf16* b,
                                       int B, int T, const float* state_pool, int pool_slots,
                                       const int32_t* state_idx, kda_bf16* o, float* snapshots,
                                       int32_t* err_flag, void* stream) {
  return verify_common(dims, gate, mixed_qkv, row_stride, a, b, B, T, nullptr, state_pool,
                       pool_slots, state_idx, o, snapshots, err_flag, stream, false);
}

extern "C" kda_status kda_verify_tree(kda_dims dims, kda_gate gate, const kda_bf16* mixed_qkv,
                                      int64_t row_stride, const kda_bf16* a, const kda_bf16* b,
                                      int B, int T, const int32_t* parent_idx,
                                      const float* state_pool, int pool_slots,
                                      const int32_t* state_idx, kda_bf16* o, float* snapshots,
                                      int32_t* err_flag, void* stream) {
  return verify_common(dims, gate, mixed_qkv, row_stride, a, b, B, T, parent_idx, state_pool,
                       pool_slots, state_idx, o, snapshots, err_flag, stream, true);
}

extern "C" kda_status kda_commit(kda_dims dims, const float* snapshots, int B, int T,
                                 const int32_t* accepted, float* state_pool, int pool_slots,
                                 const int32_t* state_idx, int32_t* err_flag, void* stream) {
  kda_status s = check_dims(dims);
  if (s != KDA_OK) return s;
  if (!state_pool || !state_idx) return KDA_ERR_NULL_ARG;
  if (B < 0 || T < 1 || pool_slots < 0) return KDA_ERR_SHAPE;
  if (B == 0) return KDA_OK;
  if (!snapshots || !accepted) return KDA_ERR_NULL_ARG;
  if (!aligned16(snapshots) || !aligned16(state_pool)) return KDA_ERR_ALIGNMENT;
  const size_t slot_elems = (size_t)dims.HV * dims.V * dims.K;
  // 16 KiB per CTA (256 threads x kCommitVec float4): a 1 MiB slot spreads
  // over 64 CTAs per request.
  const int per_slot = (int)((slot_elems / 4 + 256 * kCommitVec - 1) / (256 * kCommitVec));
  dim3 grid(per_slot, B);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  record_stage(0, st);
  commit_kernel<<<grid, 256, 0, st>>>(snapshots, T, accepted, state_pool, pool_slots, state_idx,
                                      slot_elems, err_flag);
  s = launch_status();
  record_stage(1, st);
  record_stage(2, st);
  return s;
}

extern "C" size_t kda_replay_ring_bytes(kda_dims dims, int B, int T) {
  if (B < 0 || T < 1 || dims.HV <= 0) return 0;
  return (size_t)B * T * dims.HV * kRingFloats * sizeof(float);
}

extern "C" kda_status kda_verify_chain_replay(kda_dims dims, kda_gate gate,
                                              const kda_bf16* mixed_qkv, int64_t row_stride,
                                              const kda_bf16* a, const kda_bf16* b, int B, int T,
                                              const float* state_pool, int pool_slots,
                                              const int32_t* state_idx, kda_bf16* o, float* ring,
                                              int32_t* err_flag, void* stream) {
  StepArgs args{};
  kda_status s = check_packed(dims, gate, mixed_qkv, row_stride, a, b, B, state_pool, pool_slots,
                              state_idx, o, &args);
  if (s != KDA_OK) return s;
  if (T < 1) return KDA_ERR_SHAPE;
  if (B == 0) return KDA_OK;
  if (!ring) return KDA_ERR_NULL_ARG;
  if (!aligned16(ring)) return KDA_ERR_ALIGNMENT;
  args.T = T;
  args.pool = const_cast<float*>(state_pool);  // read only in verify
  args.o = o;
  args.ring = ring;
  args.err_flag = err_flag;
  return launch_recurrent<kChainReplay>(args, static_cast<cudaStream_t>(stream));
}

extern "C" kda_status kda_commit_replay(kda_dims dims, const float* ring, int B, int T,
                                        const int32_t* accepted, float* state_pool, int pool_slots,
                                        const int32_t* state_idx, int32_t* err_flag,
                                        void* stream) {
  kda_status s = check_dims(dims);
  if (s != KDA_OK) return s;
  if (!state_pool || !state_idx) return KDA_ERR_NULL_ARG;
  if (B < 0 || T < 1 || pool_slots < 0) return KDA_ERR_SHAPE;
  if (B == 0) return KDA_OK;
  if (!ring || !accepted) return KDA_ERR_NULL_ARG;
  if (!aligned16(ring) || !aligned16(state_pool)) return KDA_ERR_ALIGNMENT;
  StepArgs args{};
  args.H = dims.H;
  args.HV = dims.HV;
  args.G = dims.HV / dims.H;  // check_dims: HV is a positive multiple of H
  args.dtype = dims.dtype;
  args.B = B;
  args.T = T;
  args.pool = state_pool;
  args.pool_slots = pool_slots;
  args.state_idx = state_idx;
  args.ring = const_cast<float*>(ring);
  args.accepted = accepted;
  args.err_flag = err_flag;
  return launch_recurrent<kCommitReplay>(args, static_cast<cudaStream_t>(stream));
}
