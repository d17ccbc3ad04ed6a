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
//   O      = scale (Qtil S0 + P U) = scale (Q' S0 + P Util),  Q' = Qtil - P W,
//            Qtil_t = q_t e^{Gam_t}
//   S_L    = Diag(e^{Gam_L}) S0 + Khat^T U,  Khat_i = k_i e^{Gam_L - Gam_i}
// Rows past the end of a sequence are q = k = v = 0, beta = 0, g = 0, which
// leave every quantity above unchanged.  Writing O through Q' = Qtil - P W
// moves the cancellation between Qtil S0 and P W S0 into the per-chunk FP32
// transform.  The chunk's end state is affine in its start state,
//   S_L = M_c S0 + B_c,  M_c = Diag(e^{Gam_L}) - Khat^T W,  B_c = Khat^T Util,
// so the sequential part of the prefill is one product per chunk.  The
// state-dependent products split both operands into BF16 hi + lo and sum
// three BF16 products (hi hi, hi lo, lo hi): with slow decay the state
// carries its errors over many chunks, and a single BF16 rounding of M_c
// (2^-9 relative) would move it by several 1e-3 of its RMS over 64 chunks.
// Q' (which only reaches o) is one BF16 operand against the split state.
//
// Decay factors inside A and P are split at a reference token r, the LAST
// token of each 16-token block of i: e^{Gam_t-Gam_i} = e^{Gam_t-Gam_r} e^{Gam_r-Gam_i}.
// The right factor is <= 1 for every i of the block.  The left factor is <= 1
// for t >= r and at most e^{15 |g|min} for the block's own earlier rows, which
// stays inside FP32 for per-token log-decays >= -5.8 (the bounded gate at
// lower bound -5 is inside that).  A left factor that underflows can only
// drop terms that are smaller still.
//
// Two kernels (a third checks given log-decays first):
//   chunk_transform_tc_kernel  persistent, one CTA per SM looping over
//                           (chunk, head) units, all chunks in parallel:
//                           rows fed by TMA, fold and cumulative decay on the
//                           CUDA cores, A and P as tcgen05 products of
//                           decay-split factors, (I+A)^-1 blocked on the CUDA
//                           cores, then W, Util, P W, P Util and the map
//                           Khat^T [W | Util] as tcgen05 products.  Writes
//                           one workspace record per (chunk, head): M_c (BF16
//                           hi/lo, only where it is not all zero) and Q' in
//                           the tensor-core operand layout, B_c and P Util in
//                           FP32, and per value slice the threshold below
//                           which M_c S cannot change an FP32 bit of S.
//   state_pass_kernel       per (sequence, head, 32 value columns) chain,
//                           sequential over the chunks, on tcgen05:
//                             S_{i+1} = M_c S_i + B_c   (left out where the
//                                       product cannot change the result)
//                             O_i     = scale (Q' S_i + P Util)
//                           with S in FP32 registers, re-split into a BF16
//                           hi/lo operand each chunk.  Long chains run as two
//                           CTAs, the second restarting behind a chunk whose
//                           product is left out whatever its start state.
#include <cuda.h>  // CUtensorMap and its enums (the encoder is fetched at run time)
#include <cudaTypedefs.h>

#include <atomic>

#include "kda_host.h"
#include "kda_tc.cuh"

namespace kda {
namespace {

constexpr int kChunk = 64;
constexpr int kLd = 132;  // padded row stride (floats) of 64 x 128 tiles in shared memory
constexpr int kLdT = 65;  // padded row stride of 64 x 64 tiles
constexpr int kVs = 32;   // value columns per state-pass CTA
constexpr int kSlices = kHeadDim / kVs;

// Workspace record of one (chunk, head), bytes.  Tiles are BF16, K-major,
// 128-byte swizzled (see kda_tc.cuh) so they can be bulk-copied straight into
// shared memory; Util and P Util are FP32 in [slice][column quad][64][4]
// order (slice = 32 value columns), so that a thread reading one token's four
// columns and its neighbours reading the next tokens touch consecutive
// 16-byte words.
constexpr uint32_t kRecM = 0;                                  // M_c hi, 128 x 128 (rows c', K = c)
constexpr uint32_t kRecML = kRecM + 128 * 128 * 2;             // M_c lo
constexpr uint32_t kRecQ = kRecML + 128 * 128 * 2;             // Q' (BF16), 64 x 128
constexpr uint32_t kRecB = kRecQ + 64 * 128 * 2;               // B_c, FP32 [slice][32 columns][128 channels]
constexpr uint32_t kRecOi = kRecB + kHeadDim * kHeadDim * 4;   // P Util, FP32 [slice][quad][64][4]
constexpr uint32_t kRecMeta = kRecOi + kChunk * kHeadDim * 4;   // FP32 [slice] {tau, ||B_c||}
constexpr uint32_t kRecBytes = kRecMeta + 128;
// Skipping a chain product.  With r = 128 max|M_c| >= every row sum of |M_c|,
// each element of the chain product M_c S is at most about r max|S| in
// magnitude (the split operands add a factor below 1 + 2^-7).  When that is
// below half an ulp of every element of B_c -- below 2^-25 min|B_c| -- the
// FP32 sum S_end = M_c S + B_c rounds to B_c whatever the product is, so the
// product can be left out without changing a bit of the state.  The record
// keeps tau = 2^-27 min|B_c| / r per value slice (a factor 4 of margin); the
// pass skips the product iff max|S| <= tau, the max taken over the slice's
// start state.  tau = +inf marks an all-zero M_c, which is not stored.
// Next to tau the record keeps ||B_c||_F of the slice, rounded up by 2^-10:
// with L2-normalised keys, beta <= 1 and g <= 0 every token's factor
// (I - beta k k^T) Diag(e^g) has norm <= 1, so M_c has too, and
// ||S_{c+1}|| <= ||S_c|| + ||B_c|| bounds every element of a later state
// before it is computed (see the pass).
constexpr float kSkipMargin = 7.450580596923828125e-09f;  // 2^-27
constexpr float kNormRoundUp = 1.0009765625f;              // 1 + 2^-10

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
  int64_t inter_chunks;       // chunk records `intermediate` holds
  uint8_t* ws;                // the (chunk, head) records
  const int32_t* seq_flags;   // [num_seqs] nonzero: sequence rejected (given decay
                              // out of range); nullptr when nothing is checked
  int32_t* err_flag;
  int64_t tx_units;  // (chunk, head) units of this transform launch
  int parts;  // CTAs (items of the state pass) per (sequence, head, slice) chain
  // Start states [num_seqs][HV][V][K] staged by the transform for a pass that
  // runs each chain in parts (nullptr: the pass reads the pool).  A later
  // part writes the pool's final state, so no part may read the slot itself.
  float* init_states;
  uint32_t* item_counter;  // the multi-item pass's claims (zeroed before the call's kernels)
};

__device__ __forceinline__ int64_t seq_begin(const PrefillArgs& a, int n) {
  return a.cu_seqlens ? (int64_t)a.cu_seqlens[n] : a.total_tokens / a.num_seqs * n;
}

// Sequences per lane per step of the warp walks below: their loads are all
// in flight at once.
constexpr int kWalkPerLane = 4;

// Checks cu_seqlens (0 .. total_tokens, non-decreasing).  A whole warp,
// 128 sequences per step; every lane gets the answer.
__device__ bool seqlens_valid_warp(const PrefillArgs& a, int lane) {
  if (!a.cu_seqlens) return true;
  if (a.cu_seqlens[0] != 0 || a.cu_seqlens[a.num_seqs] != a.total_tokens) return false;
  for (int n0 = 0; n0 < a.num_seqs; n0 += 32 * kWalkPerLane) {
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kWalkPerLane; ++i) {
      const int n = n0 + 32 * i + lane;
      bad |= n < a.num_seqs && a.cu_seqlens[n + 1] < a.cu_seqlens[n];
    }
    if (__any_sync(0xffffffffu, bad)) return false;
  }
  return true;
}

// Chunks of sequences [from, to).  A whole warp, 128 sequences per step.
__device__ int64_t chunk_count_warp(const PrefillArgs& a, int from, int to, int lane) {
  int64_t count = 0;
  for (int m0 = from; m0 < to; m0 += 32 * kWalkPerLane) {
    uint32_t c = 0u;
#pragma unroll
    for (int i = 0; i < kWalkPerLane; ++i) {
      const int m = m0 + 32 * i + lane;
      c += m < to ? (uint32_t)((seq_begin(a, m + 1) - seq_begin(a, m) + kChunk - 1) / kChunk) : 0u;
    }
    count += __reduce_add_sync(0xffffffffu, c);
  }
  return count;
}

struct ChunkLoc {
  int n;        // sequence, -1 if the chunk id is past the last chunk
  int64_t t0;   // first token of the chunk
  int len;      // tokens in the chunk (1..64)
};

// Maps sorted global chunk ids (sequence-major) to their sequences and token
// ranges: lane l resolves cid[0] and cid[1] (-1: none), ascending over
// (lane, 0) then (lane, 1) among the valid ones.  A whole warp walks the
// sequences 32 at a time (one prefix sum of their chunk counts per step) and
// stops past the largest id; each lane finds its ids' sequences among the
// step's 32 by a binary search over the lanes' first chunk ids.
__device__ void locate_chunks_warp(const PrefillArgs& a, const int64_t (&cid)[2], ChunkLoc (&out)[2], int lane) {
  out[0] = out[1] = ChunkLoc{-1, 0, 0};
  int64_t hi = cid[0] > cid[1] ? cid[0] : cid[1];
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const int64_t y = __shfl_xor_sync(0xffffffffu, hi, o);
    hi = y > hi ? y : hi;
  }
  int64_t base = 0;
  for (int m0 = 0; m0 < a.num_seqs && base <= hi; m0 += 32) {
    const int m = m0 + lane;
    const int64_t b = m < a.num_seqs ? seq_begin(a, m) : 0, e = m < a.num_seqs ? seq_begin(a, m + 1) : 0;
    const int64_t nch = (e - b + kChunk - 1) / kChunk;
    int64_t incl = nch;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int64_t lo = base + incl - nch;  // first chunk id of sequence m
    const int64_t end = base + __shfl_sync(0xffffffffu, incl, 31);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      int j = 0;  // the last lane whose first chunk id is <= cid[i]
#pragma unroll
      for (int step = 16; step; step >>= 1) {
        const int64_t lj = __shfl_sync(0xffffffffu, lo, j + step);
        if (cid[i] >= lj) j += step;
      }
      const int64_t lo_j = __shfl_sync(0xffffffffu, lo, j), b_j = __shfl_sync(0xffffffffu, b, j),
                    e_j = __shfl_sync(0xffffffffu, e, j);
      if (cid[i] >= base && cid[i] < end) {
        const int64_t t0 = b_j + (cid[i] - lo_j) * kChunk;
        out[i] = ChunkLoc{m0 + j, t0, (int)(e_j - t0 < kChunk ? e_j - t0 : kChunk)};
      }
    }
    base = end;
  }
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

// Programmatic dependent launch: the chunk transform lets the state pass be
// scheduled before it ends (its CTAs then take SMs as transform CTAs leave),
// and the pass waits here for the transform's completion and memory before
// it reads a record.  Without a dependent launch both are no-ops.
__device__ __forceinline__ void grid_dependency_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Per-chunk transform on tcgen05 (all chunks of all sequences in parallel).
//
//   M1, two products, D = L R^T with L rows [k-side; q-side] of
//        Lk_t = k_t e^{Gam_t - Gam_r},  Lq_t = q_t e^{Gam_t - Gam_r},  R_i = k_i e^{Gam_r - Gam_i}:
//     round a (M=128 N=64): rows t < 32 against r = 15 (columns 0-31, i < 32) and
//                           rows t >= 32 against r = 31 (columns 32-63, i < 32);
//     round b (M=128 N=32): rows t >= 32 against r = 47 (i >= 32).
//     Within a 32-token window every factor is bounded by e^{16 |g|min}; across
//     windows (t >= 32 > i, r = 31) both factors are <= 1.  So with per-token
//     log-decays >= -5.5 no factor leaves FP32 range; entries with i > t
//     may overflow and are masked.  Operands are TF32 (FP32 rounded to
//     nearest), one pass: A and P only shape W, Util and P Util through
//     (I+A)^-1, where an input error of 2^-11 relative stays well inside the
//     output tolerance, and the state error stays near 1e-4 of its RMS.
//   (I+A)^-1 on the CUDA cores (64 x 64, blocked 16 x 16).
//   A2 = [I; P] (I+A)^-1 on the tensor core (M=128 N=64 K=64).
//   M2: [Ti; P Ti] [beta Ktil | beta V]^T -> W | Util (rows 0-63), P W | P Util
//        (rows 64-127).  M=128 N=256 K=64.
// A2 and M2 use BF16 hi/lo splits of both operands (three MMAs each).

constexpr float kMinLogDecay = -5.5f;  // smallest per-token log-decay the windows allow
constexpr int kLdB = 136;       // padded row stride (BF16 elements) of the raw q, k, v tiles
constexpr int kTxThreads = 1024;
constexpr int kTxWarps = kTxThreads / 32;
// Tensor maps of the raw token rows, [T][heads][128] 16-bit elements, box =
// 64 tokens of one head.  The q, k, v boxes are kLdB elements wide: the 8
// elements past the row's 128 are outside the tensor and land as zeros, so
// that the box fills the padded rows of Qs, Ks, Vs exactly.
struct RowMaps {
  CUtensorMap q, k, v, g;
};
constexpr int kRowThread = 32;  // issues the row copies (thread 0 issues the products)

// 3-D tiled tensor copy global -> shared, completion on an mbarrier.  The
// shared address is 128-byte aligned; coordinates are (element, head, token).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(tc::smem_u32(bar))
      : "memory");
}
constexpr uint32_t kRowBytes = 3u * kChunk * kLdB * 2 + kChunk * kHeadDim * 2;  // one unit's four boxes

constexpr uint32_t kTxL = 0;                          // L: TF32 128 x 128
constexpr uint32_t kTxR = kTxL + 128 * 128 * 4;       // R: TF32 64 x 128
constexpr uint32_t kTxB2 = 0;                         // B2 hi, lo: 256 x 64 each (reuses L/R)
constexpr uint32_t kTxB3 = 0;                          // [W^T; Util^T] hi, lo: 256 x 64 each (reuses B2)
constexpr uint32_t kTxMs = 0;                          // M_c hi, lo output staging (reuses B3)
constexpr uint32_t kTxAf = 0;                         // A FP32 [64][kLdT] (reuses L/R)
constexpr uint32_t kTxA2 = kTxR + 2 * 64 * 128 * 2;   // A2 hi, lo: 128 x 64 each
constexpr uint32_t kTxQ = kTxA2 + 2 * 128 * 64 * 2;   // raw q BF16 [64][kLdB]
constexpr uint32_t kTxK = kTxQ + kChunk * kLdB * 2;   // raw k
constexpr uint32_t kTxV = kTxK + kChunk * kLdB * 2;   // raw v
constexpr uint32_t kTxG = kTxV + kChunk * kLdB * 2;   // Gam FP32 [64][kLd]
constexpr uint32_t kTxTf = kTxAf + kChunk * kLdT * 4;  // (I+A)^-1 FP32 [64][kLdT] (reuses L/R)
constexpr uint32_t kTxMisc = kTxG + kChunk * kLd * 4;  // rq, rk, beta [64] each + scratch [1536]
                                                       // + dt_bias [128], A_log [1] (+3),
                                                       // raw beta [64] (16-bit)
constexpr uint32_t kTxEnd = kTxMisc + (3 * kChunk + 1536 + kHeadDim + 4 + kChunk / 2) * 4;
constexpr int kDescBatch = 64;  // unit descriptors looked up together
constexpr uint32_t kTransformTcSmem = kTxEnd + 1024;
constexpr uint32_t kTxTmemCols = 512;  // M1, A2, M2: 0-255; the map product: 256-511
static_assert(kTxQ % 128 == 0 && kTxK % 128 == 0 && kTxV % 128 == 0 && (kTxA2 + 128 * 64 * 2) % 128 == 0,
              "tensor-copy destinations are 128-byte aligned");
static_assert(2 * 256 * 64 * 2 <= kTxA2, "B2 fits in the L/R region");
static_assert(kTxTf + kChunk * kLdT * 4 <= kTxR, "A and (I+A)^-1 stay below X in the R region");
static_assert(kTxB3 + 2 * 256 * 64 * 2 <= kTxR && kTxMs + 2 * 128 * 128 * 2 <= kTxR,
              "B3 and the M_c staging stay below Khat^T in the R region");
static_assert(kTxQ % 16 == 0 && kTxK % 16 == 0 && kTxV % 16 == 0 && kTxG % 16 == 0 &&
                  kTxTf % 16 == 0 && kTxMisc % 16 == 0 && kTxA2 % 1024 == 0 && kTxR % 1024 == 0,
              "alignment");
static_assert(kTransformTcSmem + kDescBatch * 16 + 256 <= 232448, "shared memory");

// Eight consecutive values -> one 16-byte chunk in each of hi and lo
// (hi = RN(x), lo = RN(x - hi), both BF16).
__device__ __forceinline__ void split8(const float* x, uint4& h, uint4& l);
__device__ __forceinline__ void st_split8(uint8_t* hi, uint8_t* lo, uint32_t off, const float* x) {
  uint4 h, l;
  split8(x, h, l);
  *reinterpret_cast<uint4*>(hi + off) = h;
  *reinterpret_cast<uint4*>(lo + off) = l;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)float_to_bf16_bits(lo) | ((uint32_t)float_to_bf16_bits(hi) << 16);
}

// Eight consecutive values -> their BF16 hi and lo parts as two 16-byte words.
__device__ __forceinline__ void split8(const float* x, uint4& h, uint4& l) {
  uint32_t hh[4], ll[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 hb = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
    const float2 hf = __bfloat1622float2(hb);
    const __nv_bfloat162 lb = __floats2bfloat162_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y);
    hh[e] = *reinterpret_cast<const uint32_t*>(&hb);
    ll[e] = *reinterpret_cast<const uint32_t*>(&lb);
  }
  h = make_uint4(hh[0], hh[1], hh[2], hh[3]);
  l = make_uint4(ll[0], ll[1], ll[2], ll[3]);
}

// Element (t, c) of a raw 16-bit input tile (BF16 or FP16 bits), widened.
template <bool F16>
__device__ __forceinline__ float in_at(const uint8_t* tile, int t, int c) {
  return in16_to_float<F16>(reinterpret_cast<const uint16_t*>(tile)[t * kLdB + c]);
}

// Four consecutive values of row t, columns [c, c+4), of a raw input tile.
template <bool F16>
__device__ __forceinline__ float4 ld_in4(const uint8_t* tile, int t, int c) {
  return in16x4_to_f4<F16>(*reinterpret_cast<const uint2*>(tile + (t * kLdB + c) * 2));
}

__device__ __forceinline__ float4 scale4(float4 a, float s) {
  return make_float4(a.x * s, a.y * s, a.z * s, a.w * s);
}

__device__ __forceinline__ float4 mul4(float4 a, float4 b) {
  return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w);
}

// e^{a - b} element-wise, for decay factors.
__device__ __forceinline__ float4 exp_diff4(float4 a, float4 b) {
  return make_float4(decay_exp(a.x - b.x), decay_exp(a.y - b.y), decay_exp(a.z - b.z),
                     decay_exp(a.w - b.w));
}

// Global chunk id of transform unit u (arithmetic only; see unit_loc).
__device__ __forceinline__ int64_t unit_cid(const PrefillArgs& a, int64_t u) { return u / a.HV; }

// Persistent: CTA b takes units b, b + gridDim.x, ...  The next unit's q, k, v
// and gate rows are copied into shared memory while this unit finishes.
template <bool F16>
__global__ void __launch_bounds__(kTxThreads, 1)
    chunk_transform_tc_kernel(const __grid_constant__ PrefillArgs a, const __grid_constant__ RowMaps rm) {
  extern __shared__ uint8_t smraw[];
  // Unit descriptor: first token and length of the unit's chunk, and whether
  // it is its sequence's first chunk; n < 0 marks a unit that is skipped (no
  // chunk, padding or rejected sequence).
  struct UnitDesc {
    int64_t t0;
    int n;
    int16_t len, first;
  };
  static_assert(sizeof(UnitDesc) == 16, "descriptor size");
  __shared__ uint64_t mma_bar;
  __shared__ uint64_t row_bar;  // a unit's q, k, v and gate input rows landed
  __shared__ uint32_t tmem_base;
  __shared__ UnitDesc s_desc[kDescBatch];
  __shared__ int s_abort, s_ok;
  __shared__ uint32_t s_mmax, s_bmin[kSlices];  // max|M_c|, min|B_c| per slice (FP32 bits, >= 0)
  __shared__ float s_bsq[kSlices];                // sum of B_c^2 per slice

  uint8_t* sb = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
  uint8_t* Lt = sb + kTxL;  // M1 left operand, TF32 128 x 128
  uint8_t* Rt = sb + kTxR;  // M1 right operand, TF32 64 x 128
  uint8_t* Rh = Rt;         // the R region, later reused for BF16 hi/lo operands
  uint8_t* Bh = sb + kTxB2;
  uint8_t* Bl = Bh + 256 * 64 * 2;
  uint8_t* A2h = sb + kTxA2;
  uint8_t* A2l = A2h + 128 * 64 * 2;
  uint8_t* Gs = A2l;  // raw gate input [64][128] (16-bit), dead from M2 to the next A2 product
  uint8_t* Qs = sb + kTxQ;
  uint8_t* Ks = sb + kTxK;
  uint8_t* Vs = sb + kTxV;
  float* GM = reinterpret_cast<float*>(sb + kTxG);
  float* Af = reinterpret_cast<float*>(sb + kTxAf);
  float* Tf = reinterpret_cast<float*>(sb + kTxTf);
  float* rq = reinterpret_cast<float*>(sb + kTxMisc);
  float* rk = rq + kChunk;
  float* bt = rk + kChunk;
  float* X = bt + kChunk;  // [6][16][16]
  float* gbias = X + 1536;    // dt_bias of the unit's head [128]
  float* galog = gbias + kHeadDim;  // A_log of the unit's head
  uint16_t* braw = reinterpret_cast<uint16_t*>(galog + 4);  // raw beta of the unit's tokens

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_dependency_launch();
  if (warp == 1) {
    const bool ok = seqlens_valid_warp(a, lane);
    if (lane == 0) {
      s_ok = ok;
      if (!ok && blockIdx.x == 0) set_error(a.err_flag, KDA_DEVERR_SEQLENS);
    }
  }
  if (tid == 0) {
    s_abort = 0;
    tc::mbar_init(&mma_bar, 1);
    tc::mbar_init(&row_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kTxTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  uint32_t phase = 0;
  // Descriptors of this CTA's next kDescBatch units (chunk-major: unit u is
  // chunk u / HV, head u % HV), by warp 0: the batch's chunk ids ascend, so
  // one walk over the sequences locates them all; then each lane checks its
  // two units' slots.
  static_assert(kDescBatch == 64, "two units per lane of warp 0");
  auto describe_batch = [&](int64_t u0) {
    int64_t cid[2];
    ChunkLoc l[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int64_t uu = u0 + (int64_t)(lane + 32 * i) * gridDim.x;
      cid[i] = uu < a.tx_units ? uu / a.HV : -1;
    }
    locate_chunks_warp(a, cid, l, lane);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      UnitDesc d{0, -1, 0, 0};
      if (l[i].n >= 0) {
        const int slot = a.state_idx[l[i].n];
        const bool live = slot >= 0 && slot < a.pool_slots &&        // else padding / rejected
                          !(a.seq_flags && a.seq_flags[l[i].n]);  // given decay out of range
        if (live) d = UnitDesc{l[i].t0, l[i].n, (int16_t)l[i].len, (int16_t)(l[i].t0 == seq_begin(a, l[i].n))};
      }
      s_desc[lane + 32 * i] = d;
    }
  };
  // A unit's raw q, k, v rows into Qs, Ks, Vs and its gate input rows into Gs
  // (one tensor copy of 64 token rows per tensor, issued by thread
  // kRowThread and completing on row_bar; rows past the last token land as
  // zeros, rows of the next sequence are zeroed after landing), dt_bias and
  // A_log of its head into gbias and galog, and the raw beta of its tokens
  // into braw (plain loads by threads 64-127, which have nothing else to do
  // until the next barrier).  Every issued batch is awaited once, at the fold
  // of its unit.
  auto issue_rows = [&](const UnitDesc& ud, int hh) {
    if (tid == kRowThread) {
      const int hkk = hh / (a.HV / a.H), t0 = (int)ud.t0;
      tc::mbar_expect_tx(&row_bar, kRowBytes);
      tc::fence_async_smem();  // the previous unit's reads of these rows come first
      tma_load_3d(Qs, &rm.q, 0, hkk, t0, &row_bar);
      tma_load_3d(Ks, &rm.k, 0, hkk, t0, &row_bar);
      tma_load_3d(Vs, &rm.v, 0, hh, t0, &row_bar);
      tma_load_3d(Gs, &rm.g, 0, hh, t0, &row_bar);
    }
    if (tid < kHeadDim / 4 && a.gate.dt_bias) cp_async16(gbias + tid * 4, a.gate.dt_bias + hh * kHeadDim + tid * 4);
    if (tid == kHeadDim / 4 && a.gate.A_log) cp_async4(galog, a.gate.A_log + hh);
    cp_async_commit();
    if (tid >= kChunk && tid < 2 * kChunk) {
      const int t = tid - kChunk;
      braw[t] = t < ud.len ? a.beta[(ud.t0 + t) * a.HV + hh] : 0;
    }
  };
  bool rows_ready = false;  // this unit's rows were copied during the previous unit
  uint32_t row_phase = 0;   // row_bar's phase of the next batch awaited
  int it = 0;               // units of this CTA so far
  for (int64_t u = blockIdx.x; s_ok && u < a.tx_units; u += gridDim.x, ++it) {
    const int bi = it % kDescBatch;
    if (bi == 0) {
      __syncthreads();  // nobody reads the previous batch any more
      if (warp == 0) describe_batch(u);
    }
    __syncthreads();  // every thread is done with the previous unit's shared values
    if (tid == 0) {  // read by 9c, after several barriers
      s_mmax = 0u;
      for (int sl = 0; sl < kSlices; ++sl) {
        s_bmin[sl] = 0x7f800000u;  // +inf
        s_bsq[sl] = 0.f;
      }
    }
    const UnitDesc ud = s_desc[bi];
    if (ud.n < 0) {
      rows_ready = false;
      continue;
    }
    const int h = (int)(u % a.HV);
    const int64_t cid = unit_cid(a, u);
    const int len = ud.len;
    const GateArgs& ga = a.gate;
    const int K = kHeadDim;
    uint8_t* rec = a.ws + ((size_t)cid * a.HV + h) * kRecBytes;

    // 1. fold.  The unit's rows are in shared memory (copied during the
    //    previous unit, or now).  Warp w owns tokens [2w, 2w+2), lane l
    //    channels [4l, 4l+4): every shared-memory access of a warp is one
    //    whole row.  Per-token norms and beta, and Gam by warp-blocked prefix:
    //    each warp's running sum (its last token's is the warp's total), warp
    //    0 turns the 32 totals into their prefix in place (in warp order, so
    //    the sums associate as a sequential scan's would), and each warp adds
    //    the total before it to its other token.  The previous
    //    unit's output staging (L/R and A2h regions) may still be read by its
    //    bulk stores: the fold writes none of it.
    if (a.init_states && ud.first) {  // the sequence's first chunk: stage its start state
      const float4* src = reinterpret_cast<const float4*>(
          a.pool + ((size_t)a.state_idx[ud.n] * a.HV + h) * kHeadDim * kHeadDim);
      float4* dst = reinterpret_cast<float4*>(a.init_states + ((size_t)ud.n * a.HV + h) * kHeadDim * kHeadDim);
      for (int i = tid; i < kHeadDim * kHeadDim / 4; i += kTxThreads) __stcg(dst + i, __ldcg(src + i));
    }
    if (!rows_ready) issue_rows(ud, h);
    cp_async_wait_all();
    if (!tc::mbar_wait(&row_bar, row_phase)) s_abort = 1;
    row_phase ^= 1;
    rows_ready = false;
    if (len < kChunk) {  // rows past the chunk's end (the next sequence's, or zeros): zero
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
      for (int i = tid; i < (kChunk - len) * 16; i += kTxThreads) {
        const int r = len + (i >> 4), p = i & 15;
        reinterpret_cast<uint4*>(Qs + r * kLdB * 2)[p] = z;
        reinterpret_cast<uint4*>(Ks + r * kLdB * 2)[p] = z;
        reinterpret_cast<uint4*>(Vs + r * kLdB * 2)[p] = z;
        reinterpret_cast<uint4*>(Gs + r * kHeadDim * 2)[p] = z;
      }
    }
    __syncthreads();
    {
      constexpr int kTpw = kChunk / kTxWarps;  // tokens per warp
      const int c = lane * 4;
      const float exp_alog = ga.A_log ? __expf(*galog) : 0.f;
      const float4 bias = ga.dt_bias ? f4(gbias + c) : make_float4(0.f, 0.f, 0.f, 0.f);
      if (tid < kChunk) bt[tid] = tid < len ? fold_beta(ga, in16_to_float<F16>(braw[tid])) : 0.f;
      float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u2 = 0; u2 < kTpw; ++u2) {
        const int t = warp * kTpw + u2;
        const bool live = t < len;
        const float4 q4 = ld_in4<F16>(Qs, t, c), k4 = ld_in4<F16>(Ks, t, c);
        const float4 a4 = in16x4_to_f4<F16>(*reinterpret_cast<const uint2*>(Gs + (t * K + c) * 2));
        const float sq = warp_sum(dot4(q4, q4)), sk = warp_sum(dot4(k4, k4));
        float4 g4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (live)
          g4 = make_float4(gate_log_decay(ga, a4.x, exp_alog, bias.x),
                           gate_log_decay(ga, a4.y, exp_alog, bias.y),
                           gate_log_decay(ga, a4.z, exp_alog, bias.z),
                           gate_log_decay(ga, a4.w, exp_alog, bias.w));
        if (lane == 0) {
          rq[t] = live ? (ga.use_qk_l2norm ? rsqrtf(sq + kNormEps) : 1.f) : 0.f;
          rk[t] = live ? (ga.use_qk_l2norm ? rsqrtf(sk + kNormEps) : 1.f) : 0.f;
        }
        run = make_float4(run.x + g4.x, run.y + g4.y, run.z + g4.z, run.w + g4.w);
        f4(GM + t * kLd + c) = run;
      }
      __syncthreads();
      if (warp == 0) {  // the warps' totals -> their inclusive prefix, in place, in warp order
        float4 acc = f4(GM + (kTpw - 1) * kLd + c);
#pragma unroll
        for (int w = 1; w < kTxWarps; ++w) {
          float4& x = f4(GM + (w * kTpw + kTpw - 1) * kLd + c);
          const float4 y = x;
          acc = make_float4(y.x + acc.x, y.y + acc.y, y.z + acc.z, y.w + acc.w);
          x = acc;
        }
      }
      __syncthreads();
      if (warp > 0) {  // the warp's other tokens: + the total of the warps before it
        const float4 pre = f4(GM + (warp * kTpw - 1) * kLd + c);
#pragma unroll
        for (int u2 = 0; u2 < kTpw - 1; ++u2) {
          float4& gg = f4(GM + (warp * kTpw + u2) * kLd + c);
          gg = make_float4(gg.x + pre.x, gg.y + pre.y, gg.z + pre.z, gg.w + pre.w);
        }
      }
    }
    // the previous unit's output staging (A2 region, upper L/R region) is
    // rewritten from step 2 on: its bulk stores must have read it by now
    if (tid == 0) tc::bulk_wait_read();
    __syncthreads();

    const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;

    // 3. M1 in two rounds (see the header of this kernel).  Warp w builds the
    //    rows of token w (round 1) or 32 + w (round 2), lane l channels
    //    [4l, 4l+4): every shared-memory access of a warp is one whole row.
    //    Round 1: L rows [Lk(t<32, r=15); Lq(t<32, r=15); Lk(t>=32, r=31);
    //             Lq(t>=32, r=31)], R rows [R(i<32, r=15); R(i<32, r=31)].
    //    Round 2: L rows [Lk(t>=32, r=47); Lq(t>=32, r=47)], R rows R(i>=32, r=47);
    //             L rows 64-127 keep round 1's values and their products are
    //             never read.
    static_assert(kTxWarps == 32, "M1 operands: one warp per token row");
    for (int round = 0; round < 2; ++round) {
      {
        const int tt = warp, c = lane * 4;
        if (round == 0) {
          const float4 g15 = f4(GM + 15 * kLd + c), g31 = f4(GM + 31 * kLd + c);
          const float4 ga = f4(GM + tt * kLd + c), gb = f4(GM + (32 + tt) * kLd + c);
          const float4 ka = scale4(ld_in4<F16>(Ks, tt, c), rk[tt]), qa = scale4(ld_in4<F16>(Qs, tt, c), rq[tt]);
          const float4 kb = scale4(ld_in4<F16>(Ks, 32 + tt, c), rk[32 + tt]);
          const float4 qb = scale4(ld_in4<F16>(Qs, 32 + tt, c), rq[32 + tt]);
          const float4 fa = exp_diff4(ga, g15), fb = exp_diff4(gb, g31);
          tc::st_tf32x4(Lt, tt, c, 128, mul4(ka, fa));
          tc::st_tf32x4(Lt, 32 + tt, c, 128, mul4(qa, fa));
          tc::st_tf32x4(Lt, 64 + tt, c, 128, mul4(kb, fb));
          tc::st_tf32x4(Lt, 96 + tt, c, 128, mul4(qb, fb));
          tc::st_tf32x4(Rt, tt, c, 64, mul4(ka, exp_diff4(g15, ga)));
          tc::st_tf32x4(Rt, 32 + tt, c, 64, mul4(ka, exp_diff4(g31, ga)));
        } else {
          const int t = 32 + tt;
          const float4 g47 = f4(GM + 47 * kLd + c), gt = f4(GM + t * kLd + c);
          const float4 kt = scale4(ld_in4<F16>(Ks, t, c), rk[t]), qt = scale4(ld_in4<F16>(Qs, t, c), rq[t]);
          const float4 f = exp_diff4(gt, g47);
          tc::st_tf32x4(Lt, tt, c, 128, mul4(kt, f));
          tc::st_tf32x4(Lt, 32 + tt, c, 128, mul4(qt, f));
          tc::st_tf32x4(Rt, tt, c, 32, mul4(kt, exp_diff4(g47, gt)));
        }
      }
      const int nR = round == 0 ? 64 : 32;
      tc::fence_async_smem();
      tc::tc_fence_before();
      __syncthreads();
      if (tid == 0 && !s_abort) {
        tc::tc_fence_after();
        const uint32_t idesc = round == 0 ? tc::idesc_tf32_f32(128, 64) : tc::idesc_tf32_f32(128, 32);
        const uint32_t la = tc::smem_u32(Lt), ra = tc::smem_u32(Rt);
#pragma unroll
        for (int k = 0; k < 16; ++k) {  // K = 128 in steps of 8 (32 bytes of each row)
          const uint32_t koff = (k & 3) * 32;
          tc::mma_tf32(tmem + round * 64, tc::sw128_desc(la + (k >> 2) * (128 * 128) + koff),
                       tc::sw128_desc(ra + (k >> 2) * (nR * 128) + koff), idesc, k > 0);
        }
        tc::mma_commit(&mma_bar);
      }
      if (!tc::mbar_wait(&mma_bar, phase)) s_abort = 1;
      phase ^= 1;
      tc::tc_fence_after();
    }

    // 4. A (beta-scaled, strictly lower) to FP32 for the inverse, and P (lower)
    //    straight into the A2 product's left operand X = [I; P] (128 x 64, BF16
    //    hi/lo, in the R region, dead since M1 completed).  TMEM columns:
    //    0-31  rows 0-63   : t = row & 31 (< 32),  i = col        (k rows 0-31, q rows 32-63)
    //    32-63 rows 64-127 : t = 32 + (row & 31),  i = col - 32
    //    64-95 rows 0-63   : t = 32 + (row & 31),  i = 32 + col - 64
    //    The inverse reads only A's lower blocks.  Warp groups 3-7 (640 threads)
    //    write X's identity rows (64 rows x 8 chunks) and P's zero block
    //    t < 32 <= i (32 rows x 4 chunks), one 8-column chunk each.
    uint8_t* Xh = Rh;  // X = [I; P]: 128 x 64, 16 KB each half
    uint8_t* Xl = Xh + 128 * 64 * 2;
    {
      const int wg = warp >> 2, row = (warp & 3) * 32 + lane;
      if (wg < 3) {
        float d[32];
        tc::tmem_ld16(tmem + lane_addr + wg * 32, *reinterpret_cast<float(*)[16]>(d));
        tc::tmem_ld16(tmem + lane_addr + wg * 32 + 16, *reinterpret_cast<float(*)[16]>(d + 16));
        const bool use = wg == 1 ? row >= 64 : row < 64;
        if (use) {
          const int t = (wg == 0 ? 0 : 32) + (row & 31);
          const int i0 = wg == 2 ? 32 : 0;
          if ((row & 63) >= 32) {  // P row t
#pragma unroll
            for (int e = 0; e < 32; ++e) d[e] = i0 + e <= t ? d[e] : 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) st_split8(Xh, Xl, tc::sw128_offset(kChunk + t, i0 + 8 * j, 128), d + 8 * j);
          } else {  // A row t
            float* dst = Af + t * kLdT + i0;
#pragma unroll
            for (int e = 0; e < 32; ++e) dst[e] = i0 + e < t ? bt[t] * d[e] : 0.f;
          }
        }
      } else {
        const int idx = tid - 384;  // 0 .. 639
        float x[8];
        if (idx < kChunk * 8) {  // identity row r, chunk ch
          const int r = idx >> 3, ch = idx & 7;
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = ch * 8 + e == r ? 1.f : 0.f;
          st_split8(Xh, Xl, tc::sw128_offset(r, ch * 8, 128), x);
        } else {  // P row t < 32, chunk 4 + ch: columns i >= 32
          const int t = (idx - kChunk * 8) >> 2, ch = 4 + ((idx - kChunk * 8) & 3);
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.f;
          st_split8(Xh, Xl, tc::sw128_offset(kChunk + t, ch * 8, 128), x);
        }
      }
      static_assert(kTxThreads - 384 == kChunk * 8 + 32 * 4, "one X chunk per thread of warp groups 3-7");
    }
    tc::tc_fence_before();
    __syncthreads();

    // 5. (I + A)^-1 = Ti, blocked in 16 x 16.  With T_ii the inverses of the
    //    diagonal blocks I + A_ii and M_ik = T_ii A_ik (k < i), block forward
    //    substitution gives T_ij = -sum_{k=j}^{i-1} M_ik T_kj, one block
    //    diagonal d = i - j at a time.
    //    5a. T_ii by forward substitution (one column per thread, threads 0-63);
    //        the other threads zero the strictly upper blocks.
    if (tid < kChunk) {
      const int b0 = (tid >> 4) * 16, col = tid & 15;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = r == col ? 1.f : 0.f;
#pragma unroll
        for (int s2 = 0; s2 < r; ++s2) acc -= Af[(b0 + r) * kLdT + b0 + s2] * x[s2];
        x[r] = acc;
        Tf[(b0 + r) * kLdT + b0 + col] = acc;
      }
    } else {
      for (int idx = tid - kChunk; idx < 6 * 256; idx += kTxThreads - kChunk) {
        const int blk = idx >> 8, r = (idx >> 4) & 15, cc = idx & 15;
        const int bi = blk < 3 ? 0 : (blk < 5 ? 1 : 2);               // (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
        const int bj = blk < 3 ? blk + 1 : (blk < 5 ? blk - 1 : 3);
        Tf[(bi * 16 + r) * kLdT + bj * 16 + cc] = 0.f;
      }
    }
    __syncthreads();
    //    5b. M_ik for the six blocks k < i, stored transposed (X[blk][m][r] =
    //        M_ik[r][m], blk = i(i-1)/2 + k).  64 threads per block, each a
    //        2 x 2 patch (rows r0, r0+1; columns c0, c0+1).
    if (tid < 6 * 64) {
      const int blk = tid >> 6, r0 = ((tid & 63) >> 3) * 2, c0 = (tid & 7) * 2;
      const int bi = blk < 1 ? 1 : (blk < 3 ? 2 : 3);
      const int bk = blk - bi * (bi - 1) / 2;
      const float* Ti0 = Tf + (bi * 16 + r0) * kLdT + bi * 16;
      const float* Ab = Af + (bi * 16) * kLdT + bk * 16 + c0;
      float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
#pragma unroll
      for (int m = 0; m < 16; ++m) {
        const float t0 = Ti0[m], t1 = Ti0[kLdT + m];
        const float b0 = Ab[m * kLdT], b1 = Ab[m * kLdT + 1];
        a00 += t0 * b0; a01 += t0 * b1; a10 += t1 * b0; a11 += t1 * b1;
      }
      float* Mt = X + blk * 256;
      *reinterpret_cast<float2*>(Mt + c0 * 16 + r0) = make_float2(a00, a10);
      *reinterpret_cast<float2*>(Mt + (c0 + 1) * 16 + r0) = make_float2(a01, a11);
    }
    __syncthreads();
    //    5c. block diagonals d = 1, 2, 3, same patches
    for (int d = 1; d < 4; ++d) {
      if (tid < (4 - d) * 64) {
        const int bj = tid >> 6, r0 = ((tid & 63) >> 3) * 2, c0 = (tid & 7) * 2;
        const int bi = bj + d;
        float a00 = 0.f, a01 = 0.f, a10 = 0.f, a11 = 0.f;
        for (int bk = bj; bk < bi; ++bk) {
          const float* Mt = X + (bi * (bi - 1) / 2 + bk) * 256 + r0;
          const float* Tk = Tf + (bk * 16) * kLdT + bj * 16 + c0;
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const float2 mm = *reinterpret_cast<const float2*>(Mt + m * 16);
            const float b0 = Tk[m * kLdT], b1 = Tk[m * kLdT + 1];
            a00 += mm.x * b0; a01 += mm.x * b1; a10 += mm.y * b0; a11 += mm.y * b1;
          }
        }
        float* dst = Tf + (bi * 16 + r0) * kLdT + bj * 16 + c0;
        dst[0] = -a00; dst[1] = -a01; dst[kLdT] = -a10; dst[kLdT + 1] = -a11;
      }
      __syncthreads();
    }

    // 6. A2 = [Ti; P Ti] on the tensor core: D = [I; P] Ti, M=128 N=64 K=64.
    //    Operands: X = [I; P] (128 x 64, K = i, written in step 4) in the R
    //    region, Ti^T (64 x 64, rows j, K = i) in the A2 region; both hi/lo.
    //    While the product runs, B2 (step 7) is built in the lower L/R region,
    //    dead by then; the result lands in TMEM columns 128-191 and is split
    //    into A2 (hi/lo) by all warps.
    {
      uint8_t* Th = A2h;                    // 64 x 64, 8 KB each half
      uint8_t* Tl = Th + 64 * 64 * 2;
      static_assert(kTxB2 + 2 * 256 * 64 * 2 <= kTxR, "B2 stays clear of X");
      if (tid < 64 * 8) {                   // Ti^T rows j
        const int j = tid >> 3, ch = tid & 7;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = Tf[(ch * 8 + e) * kLdT + j];
        st_split8(Th, Tl, tc::sw128_offset(j, ch * 8, 64), x);
      }
      tc::fence_async_smem();
      tc::tc_fence_before();
      __syncthreads();
      if (tid == 0 && !s_abort) {
        tc::tc_fence_after();
        constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 64);
        const uint32_t ah[3] = {tc::smem_u32(Xh), tc::smem_u32(Xh), tc::smem_u32(Xl)};
        const uint32_t bh[3] = {tc::smem_u32(Th), tc::smem_u32(Tl), tc::smem_u32(Th)};
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_bf16(tmem + 128, tc::sw128_desc(ah[p] + k * 32), tc::sw128_desc(bh[p] + k * 32),
                         idesc, p > 0 || k > 0);
        tc::mma_commit(&mma_bar);
      }
      // 7. B2 = [(beta Ktil)^T ; (beta V)^T] (hi/lo, swizzled 256 x 64): row -> channel
      for (int idx = tid; idx < K * 8; idx += kTxThreads) {  // rows 0-127: beta_i k-hat_i e^{Gam_i}
        const int c = idx & (K - 1), ch = idx >> 7;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int i = ch * 8 + e;
          x[e] = in_at<F16>(Ks, i, c) * (bt[i] * rk[i]) * decay_exp(GM[i * kLd + c]);
        }
        st_split8(Bh, Bl, tc::sw128_offset(c, ch * 8, 256), x);
      }
      for (int idx = tid; idx < K * 8; idx += kTxThreads) {  // rows 128-255: beta_i v_i
        const int c = idx & (K - 1), ch = idx >> 7;
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int i = ch * 8 + e;
          x[e] = in_at<F16>(Vs, i, c) * bt[i];
        }
        st_split8(Bh, Bl, tc::sw128_offset(K + c, ch * 8, 256), x);
      }
      if (!tc::mbar_wait(&mma_bar, phase)) s_abort = 1;
      phase ^= 1;
      tc::tc_fence_after();
      // TMEM -> A2 (Ti^T is dead now): warp group g takes 8 of the 64 columns
      {
        const int row = (warp & 3) * 32 + lane, c0 = (warp >> 2) * (64 / (kTxWarps / 4));
        for (int cc = 0; cc < 64 / (kTxWarps / 4); cc += 8) {
          float d[8];
          tc::tmem_ld8(tmem + lane_addr + 128 + c0 + cc, d);
          st_split8(A2h, A2l, tc::sw128_offset(row, c0 + cc, 128), d);
        }
      }
    }
    tc::fence_async_smem();
    tc::tc_fence_before();
    __syncthreads();

    // 8. M2: D = A2 B2^T, M=128 N=256 K=64
    if (tid == 0 && !s_abort) {
      tc::tc_fence_after();
      constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 256);
      const uint32_t ah[3] = {tc::smem_u32(A2h), tc::smem_u32(A2h), tc::smem_u32(A2l)};
      const uint32_t bh[3] = {tc::smem_u32(Bh), tc::smem_u32(Bl), tc::smem_u32(Bh)};
#pragma unroll
      for (int p = 0; p < 3; ++p)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          tc::mma_bf16(tmem, tc::sw128_desc(ah[p] + k * 32), tc::sw128_desc(bh[p] + k * 32), idesc,
                       p > 0 || k > 0);
      tc::mma_commit(&mma_bar);
    }
    // Khat^T (hi/lo, swizzled 128 x 64: rows c, K = token i) for the map
    // product of step 9, built in the R region (X is dead since the A2
    // product) while the tensor core runs M2.
    uint8_t* KTh = sb + kTxR;
    uint8_t* KTl = KTh + 128 * 64 * 2;
    {
      const int c = tid & (K - 1), j = tid >> 7;  // channel c, tokens [8j, 8j+8)
      static_assert(kTxThreads == kHeadDim * 8, "one Khat^T chunk per thread");
      const float gl = GM[(kChunk - 1) * kLd + c];
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int t = j * 8 + e;
        x[e] = in_at<F16>(Ks, t, c) * rk[t] * decay_exp(gl - GM[t * kLd + c]);
      }
      st_split8(KTh, KTl, tc::sw128_offset(c, j * 8, K), x);
    }
    if (!tc::mbar_wait(&mma_bar, phase)) s_abort = 1;
    phase ^= 1;
    tc::tc_fence_after();

    // 9. epilogue.  Thread (TMEM lane quadrant warp & 3, column group warp >> 2)
    //    takes lane 32 (warp & 3) + lane and 32 consecutive columns.  After M2,
    //    columns 0-127 hold W (lanes 0-63, token t = lane) | P W (lanes 64-127,
    //    t = lane - 64) and columns 128-255 Util | P Util.  M2 has finished
    //    reading its operands.
    //    9a. Q' = Qtil - P W in BF16 (a 64 x 128 tile) staged in the A2 region
    //        and bulk-stored; P Util straight to the record;
    //        W and Util written transposed (rows = channel / value column, K =
    //        token) and split into B3 = [W^T; Util^T] in the B2 region.
    //    9b. The chunk's affine map S_end = M_c S0 + B_c as one product
    //        Khat^T [W | Util] (M=128 N=256 K=64, BF16 x3) into TMEM columns
    //        256-511: M_c = Diag(gamma) - Khat^T W, B_c = Khat^T Util.
    //    9c. M_c split hi/lo, staged in the (now dead) B3 region and
    //        bulk-stored; B_c FP32 straight to the record.
    uint8_t* B3h = sb + kTxB3;
    uint8_t* B3l = B3h + 256 * 64 * 2;
    uint8_t* QQ = A2h;  // Q': 64 x 128 BF16, 16 KB
    {
      const int row = (warp & 3) * 32 + lane, cg = warp >> 2;
      uint32_t raw[2][16];
      tc::tmem_ld16_async(tmem + lane_addr + cg * 32, raw[0]);
      tc::tmem_ld16_async(tmem + lane_addr + cg * 32 + 16, raw[1]);
      tc::tmem_wait_ld();
      float d[32];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        d[e] = __uint_as_float(raw[0][e]);
        d[16 + e] = __uint_as_float(raw[1][e]);
      }
      if (row < kChunk) {  // W / Util of token t: row n = 32 cg + e of B3, column t
        const int t = row;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          uint16_t hi, lo;
          tc::split_bf16(d[e], hi, lo);
          const uint32_t off = tc::sw128_offset(cg * 32 + e, t, 256);
          *reinterpret_cast<uint16_t*>(B3h + off) = hi;
          *reinterpret_cast<uint16_t*>(B3l + off) = lo;
        }
      } else if (cg < 4) {  // Q' = Qtil - P W, channels [32 cg, 32 cg + 32) of token t
        const int t = row - kChunk, c0 = cg * 32;
        const float nq = rq[t];
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 qq = scale4(ld_in4<F16>(Qs, t, c0 + e), nq);
          const float4 gg = f4(GM + t * kLd + c0 + e);
          d[e] = qq.x * decay_exp(gg.x) - d[e];
          d[e + 1] = qq.y * decay_exp(gg.y) - d[e + 1];
          d[e + 2] = qq.z * decay_exp(gg.z) - d[e + 2];
          d[e + 3] = qq.w * decay_exp(gg.w) - d[e + 3];
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float* xs = d + 8 * j;
          *reinterpret_cast<uint4*>(QQ + tc::sw128_offset(t, c0 + 8 * j, kChunk)) =
              make_uint4(pack_bf16x2(xs[0], xs[1]), pack_bf16x2(xs[2], xs[3]), pack_bf16x2(xs[4], xs[5]),
                         pack_bf16x2(xs[6], xs[7]));
        }
      } else {  // P Util, value slice cg - 4 of token t -> [slice][quad][64][4]
        const int t = row - kChunk;
        float4* dst = reinterpret_cast<float4*>(rec + kRecOi) + (cg - 4) * (kVs / 4) * kChunk + t;
#pragma unroll
        for (int qd = 0; qd < kVs / 4; ++qd)
          dst[qd * kChunk] = make_float4(d[4 * qd], d[4 * qd + 1], d[4 * qd + 2], d[4 * qd + 3]);
      }
    }
    tc::fence_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      tc::bulk_s2g(rec + kRecQ, QQ, kChunk * 128 * 2);
      tc::bulk_commit();  // awaited at the end of the next unit's fold, or on exit
      if (!s_abort) {
        tc::tc_fence_after();
        constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 256);
        const uint32_t ah[3] = {tc::smem_u32(KTh), tc::smem_u32(KTh), tc::smem_u32(KTl)};
        const uint32_t bh[3] = {tc::smem_u32(B3h), tc::smem_u32(B3l), tc::smem_u32(B3h)};
#pragma unroll
        for (int p = 0; p < 3; ++p)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            tc::mma_bf16(tmem + 256, tc::sw128_desc(ah[p] + k * 32), tc::sw128_desc(bh[p] + k * 32),
                         idesc, p > 0 || k > 0);
        tc::mma_commit(&mma_bar);
      }
    }
    // The next unit's rows: this unit reads Qs, Ks, Vs and Gs no more, so they
    // are copied now, behind the map product's issue, and land while it and
    // 9c run.  A next unit in the next descriptor batch, or skipped, is not
    // prefetched.
    rows_ready = false;
    if (bi + 1 < kDescBatch) {
      const UnitDesc nd = s_desc[bi + 1];
      if (nd.n >= 0) {
        issue_rows(nd, (int)((u + gridDim.x) % a.HV));
        rows_ready = true;
      }
    }
    if (!tc::mbar_wait(&mma_bar, phase)) s_abort = 1;
    phase ^= 1;
    tc::tc_fence_after();
    {  // 9c: lane = output row c'
      const int row = (warp & 3) * 32 + lane, cg = warp >> 2;
      uint32_t raw[2][16];
      tc::tmem_ld16_async(tmem + lane_addr + 256 + cg * 32, raw[0]);
      tc::tmem_ld16_async(tmem + lane_addr + 256 + cg * 32 + 16, raw[1]);
      tc::tmem_wait_ld();
      float d[32];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        d[e] = __uint_as_float(raw[0][e]);
        d[16 + e] = __uint_as_float(raw[1][e]);
      }
      if (cg < 4) {  // M_c[c'][c] = gamma_c' [c == c'] - (Khat^T W)[c'][c]
        const int c0 = cg * 32;
        const float gam = decay_exp(GM[(kChunk - 1) * kLd + row]);
#pragma unroll
        for (int e = 0; e < 32; ++e) d[e] = (c0 + e == row ? gam : 0.f) - d[e];
        uint32_t mx = 0u;  // max |d| as FP32 bits (monotone for non-negative values; NaN is largest)
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = max(mx, __float_as_uint(d[e]) & 0x7fffffffu);
#pragma unroll
        for (int m = 16; m; m >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, m));
        if (lane == 0) atomicMax(&s_mmax, mx);
        uint8_t* Mh = sb + kTxMs;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          st_split8(Mh, Mh + 128 * 128 * 2, tc::sw128_offset(row, c0 + 8 * j, 128), d + 8 * j);
      } else {  // B_c, value slice cg - 4 of row c' -> [slice][value column][128 channels]
        float* dst = reinterpret_cast<float*>(rec + kRecB) + (size_t)(cg - 4) * kVs * kHeadDim + row;
#pragma unroll
        for (int e = 0; e < kVs; ++e) dst[e * kHeadDim] = d[e];  // a warp: 128 consecutive bytes
        uint32_t mn = 0xffffffffu;  // min |B_c| of the slice as FP32 bits
#pragma unroll
        for (int e = 0; e < 32; ++e) mn = min(mn, __float_as_uint(d[e]) & 0x7fffffffu);
#pragma unroll
        for (int m = 16; m; m >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, m));
        float sq = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) sq += d[e] * d[e];
        sq = warp_sum(sq);
        if (lane == 0) {
          atomicMin(&s_bmin[cg - 4], mn);
          atomicAdd(&s_bsq[cg - 4], sq);
        }
      }
    }
    if (s_abort && tid == 0) set_error(a.err_flag, KDA_DEVERR_TIMEOUT);
    tc::fence_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
      const float mmax = __uint_as_float(s_mmax);
      const float r = 128.f * mmax;  // NaN stays NaN: never skipped
      float* meta = reinterpret_cast<float*>(rec + kRecMeta);
      // an infinite or NaN bound never skips; a finite one stays below +inf,
      // which marks the all-zero map alone
      for (int sl = 0; sl < kSlices; ++sl) {
        meta[2 * sl] = s_mmax == 0u ? __int_as_float(0x7f800000)
                     : r < __int_as_float(0x7f800000) ? fminf(kSkipMargin * __uint_as_float(s_bmin[sl]) / r, 3.402823466e38f)
                                                      : -1.f;
        meta[2 * sl + 1] = sqrtf(s_bsq[sl]) * kNormRoundUp;
      }
      if (s_mmax != 0u) {  // an all-zero M_c is never read
        static_assert(kRecML == kRecM + 128 * 128 * 2, "M_c hi and lo are contiguous");
        tc::bulk_s2g(rec + kRecM, sb + kTxMs, 2 * 128 * 128 * 2);
        tc::bulk_commit();  // awaited at the end of the next unit's fold, or on exit
      }
    }
  }  // units
  cp_async_wait_all();  // no copy into shared memory outlives the CTA
  if (rows_ready) tc::mbar_wait(&row_bar, row_phase, 1u << 20);
  if (tid == 0) tc::bulk_wait_read();  // shared memory stays valid until read
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTxTmemCols);
}

// ---------------------------------------------------------------------------
// Sequential state pass on tcgen05.

// Shared-memory layout of the state pass (bytes from a 1024-aligned base).
// A stage holds one chunk's operand tiles, bulk-copied from its record in two
// parts: M_c (hi, lo), read by the chain product, and Q', read by the output
// product, each reloaded as soon as its own reader is done.  B_c and P Util go
// straight from the record into registers.
constexpr uint32_t kStM = 0;                           // M_c hi, lo: 128 x 128 each
constexpr uint32_t kStMBytes = 2 * 128 * 128 * 2;
constexpr uint32_t kStQ = kStM + kStMBytes;            // Q': 64 x 128 (two 8 KB atom columns)
constexpr uint32_t kStQBytes = kChunk * 128 * 2;
constexpr uint32_t kStageBytes = kStQ + kStQBytes;
constexpr int kSBufs = 3;                              // state operand buffers
constexpr uint32_t kSmS = 2 * kStageBytes;             // [S_hi; S_lo]^T: 64 x 128, kSBufs buffers
constexpr uint32_t kSmSBytes = 2 * kVs * kHeadDim * 2;
constexpr uint32_t kPassSmem = kSmS + kSBufs * kSmSBytes + 1024;  // + alignment slack
// TMEM: the chain product in columns 0-63 (S_hi | S_lo halves), the output
// product in 64-127 or 128-191 (two buffers)
constexpr uint32_t kTmemCols = 256;
constexpr int kOBufs = 3;  // output product buffers (TMEM columns, o_bar barriers)
static_assert(kStQ == kStM + kStMBytes && kRecQ == kRecM + kStMBytes, "the record's tiles in stage order");
static_assert(kPassSmem <= 232448, "shared memory");
// The output product is M = 64: its accumulator rows 16 q + l sit in TMEM
// lanes 32 q + l (l < 16) of the four lane quadrants.

// Copies as 16 KB pieces, which the copy engine keeps in flight together.
constexpr uint32_t kCopyPiece = 16 * 1024;
static_assert(kStMBytes % kCopyPiece == 0 && kStQBytes % kCopyPiece == 0, "whole pieces");
__device__ __forceinline__ void issue_copy(uint8_t* dst, const uint8_t* src, uint32_t bytes, uint64_t* bar) {
  tc::mbar_expect_tx(bar, bytes);
  for (uint32_t off = 0; off < bytes; off += kCopyPiece) tc::bulk_g2s(dst + off, src + off, kCopyPiece, bar);
}

// Chunks ahead of the copies whose records are prefetched into L2.
constexpr int kPassL2Ahead = 3;

// With more pass items than SMs, chains run in two parts where the sequences
// average this many tokens or more (shorter ones would mostly add items).
constexpr int64_t kMultiPartTokens = 1024;

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

constexpr int kPassEpiThreads = 512;                // 4 warps per TMEM lane quadrant
constexpr int kPassThreads = kPassEpiThreads + 64;  // + the MMA warp and the copy warp
constexpr int kColsPerThread = kVs / 4;

// Per (sequence, head, 32 value columns), sequential over the sequence's
// chunks; the 16 epilogue warps own the slice of the state.  Per chunk i,
// with S_i its start state:
//   chain   D_ch = M_hi [S_hi | S_lo] + M_lo S_hi      (M=128 N=64, then N=32)
//           S_{i+1} = D_ch[S_hi half] + D_ch[S_lo half] + B_c
//   output  D_O  = Q' [S_hi | S_lo]                     (M=64 N=64)
//           O    = scale (D_O[S_hi half] + D_O[S_lo half] + P Util)
// Warp 16 issues the products as soon as S_i's operand is written: chunk i's
// chain product, then its output product, which runs while the epilogue
// warps turn the chain product into S_{i+1}.  The epilogue finishes chunk
// i's output one chunk later (after writing S_{i+2}'s operand), so that it
// never waits for a product just issued: the output has three TMEM buffers,
// and the state operand three (chunk i's output product may still read S_i
// while S_{i+1} and S_{i+2} are written).  Warp 17 issues the stage copies
// and L2 prefetches.  Neither blocks the epilogue warps.
// kMulti: a CTA may run several items (more items than SMs); without it each
// CTA runs one, and the counters carried between items fold away.
template <bool F16, bool kMulti>
__global__ void __launch_bounds__(kPassThreads, 1) state_pass_kernel(const PrefillArgs a) {
  extern __shared__ uint8_t smraw[];
  // M_c stage j & 1 holds the j-th M_c copied (maps that are all zero are not
  // copied); Q' stage i & 1 holds chunk i's Q'.
  __shared__ uint64_t m_full[2], q_full[2];
  __shared__ uint64_t m_free[2];             // the M_c stage is free again
  __shared__ uint64_t ch_bar, o_bar[kOBufs];  // chain product done; chunk i's output product done (i % 3)
  __shared__ uint64_t s_ready[kSBufs];       // state operand buffer b written (per-warp arrivals)
  __shared__ uint32_t s_pmax[kSBufs][kPassEpiThreads / 32];  // per-warp max|S| (FP32 bits) of buffer b's state
  __shared__ uint32_t tmem_base;
  __shared__ int64_t s_t0, s_t1, s_cbase;
  __shared__ int s_state, s_abort, s_cs, s_valid;
  // counters of single roles that run on across items (see below)
  __shared__ int s_m_issued, s_q_issued, s_m_used, s_wb_n;
  __shared__ int64_t s_wb_base, s_item;
  __shared__ float s_bnd0, s_pn[kPassEpiThreads / 32];  // run start bound; per-warp sums

  uint8_t* smb = smraw + ((1024u - (tc::smem_u32(smraw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool mma_warp = warp == kPassEpiThreads / 32, copy_warp = warp == kPassEpiThreads / 32 + 1;
  const int quad = warp & 3, cg = (warp >> 2) & 3;  // TMEM lane quadrant, column group
  const int row = quad * 32 + lane;                 // key channel c (chain) or output row
  const int j0 = cg * kColsPerThread;               // first of this thread's value columns
  const int HV = a.HV, K = kHeadDim, V = kHeadDim;
  const int parts = a.parts;  // CTAs per chain
  const int64_t n_items = (int64_t)kSlices * parts * HV * a.num_seqs;

  // Once per CTA: the cu_seqlens check, the barriers and TMEM.
  if (warp == 0) {
    const bool valid = seqlens_valid_warp(a, lane);
    if (lane == 0) {
      s_valid = valid;
      s_abort = 0;
      s_m_issued = s_q_issued = s_m_used = s_wb_n = 0;
      s_wb_base = 0;
      if (!valid && blockIdx.x == 0) set_error(a.err_flag, KDA_DEVERR_SEQLENS);
      for (int i = 0; i < 2; ++i) {
        tc::mbar_init(&m_full[i], 1);
        tc::mbar_init(&q_full[i], 1);
        tc::mbar_init(&m_free[i], 1);
      }
      tc::mbar_init(&ch_bar, 1);
      for (int b = 0; b < kOBufs; ++b) tc::mbar_init(&o_bar[b], 1);
      for (int b = 0; b < kSBufs; ++b) tc::mbar_init(&s_ready[b], kPassEpiThreads / 32);  // one arrival per epilogue warp
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
  }
  if (warp == 0) tc::tmem_alloc(&tmem_base, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t dch = tmem;
  constexpr uint32_t idesc2 = tc::idesc_bf16_f32(128, 2 * kVs);
  constexpr uint32_t idesc1 = tc::idesc_bf16_f32(128, kVs);
  constexpr uint32_t idescO = tc::idesc_bf16_f32(kChunk, 2 * kVs);
  const int c = row;
  // Epilogue threads hold the state in one of two ownerships, the same for
  // the whole CTA: by channel (S[c][v0 + j0 .. + 8), c = the thread's TMEM
  // lane), which a chain product's accumulator needs, or by column
  // (S[cc0 .. + 8)[v0 + jc]), which writes the state operand with two 16-byte
  // stores instead of sixteen 2-byte ones.  A chunk whose product is
  // certainly left out (S_{i+1} = B_c) takes the second.
  float S[kColsPerThread] = {};
  bool scol = true;  // S is held by column
  const int jc = tid >> 4, cc0 = (tid & 15) * 8;
  // Counters that run on across the CTA's items, so that ring positions and
  // barrier phases continue from one item to the next: the chunks run before
  // the current item (every role; chunk ci of an item is the CTA's chunk
  // g0 + ci), the chain products waited for (epilogue), and in shared memory
  // the M_c and Q' copies issued (copy warp), the M_c stages taken (MMA warp)
  // and the chunks of sequences [0, s_wb_n), s_wb_base (warp 0).
  int g0 = 0;
  int nchain = 0;
  // Items (sequence n, head h, part, 32-column slice), slices fastest.  One
  // CTA per item where they fit the SMs; otherwise each CTA runs several,
  // which saves the set-up per item for many short sequences: CTA b takes
  // item b first, then claims the next unclaimed one from a counter whenever
  // it is free, so that chains of different lengths spread over the CTAs.
  // A CTA's claims ascend, and so do its sequences.
  auto next_item = [&]() -> int64_t {
    if constexpr (!kMulti) {
      return n_items;
    } else {
      if (tid == 0) s_item = (int64_t)gridDim.x + atomicAdd(a.item_counter, 1u);
      __syncthreads();  // rewritten only after the next item's barriers
      return s_item;
    }
  };
  for (int64_t item = blockIdx.x; s_valid && item < n_items; item = next_item()) {
    const int slice = (int)(item % kSlices), v0 = slice * kVs;
    const int64_t rest = item / kSlices;
    const int part = (int)(rest % parts), h = (int)(rest / parts % HV), n = (int)(rest / parts / HV);
    const bool reporter = slice == 0 && part == 0;
    __syncthreads();  // every thread is done with the previous item's shared values
    if (warp == 0) {  // the chunks before sequence n (on from the previous item's), and the checks
      const int64_t base = s_wb_base + chunk_count_warp(a, s_wb_n, n, lane);
      __syncwarp();
      if (lane == 0) {
        s_wb_base = base;
        s_wb_n = n;
        s_cbase = base;
        s_state = 0;
        const int slot = a.state_idx[n];
        if (slot < -1 || slot >= a.pool_slots) {
          s_state = 2;
          if (reporter && h == 0) set_error(a.err_flag, KDA_DEVERR_SLOT);
        } else if (slot == -1) {
          s_state = 1;
        } else if (a.seq_flags && a.seq_flags[n]) {
          s_state = 2;  // given log-decay out of range: flagged by decay_check_kernel
        }
        s_t0 = seq_begin(a, n);
        s_t1 = seq_begin(a, n + 1);
      }
    }
    __syncthreads();
    if (s_abort) break;
    if (s_state == 2) continue;
    const int64_t t0 = s_t0, t1 = s_t1;
    const int nch = (int)((t1 - t0 + kChunk - 1) / kChunk);  // chunks of the sequence
    // this item's share of them: its outputs and chunk-start states, and the
    // final state for the last part
    const int own0 = (int)((int64_t)part * nch / parts), own1 = (int)((int64_t)(part + 1) * nch / parts);
    if (s_state == 1) {  // padding sequence: zero outputs
      const int64_t ta = t0 + (int64_t)own0 * kChunk;
      const int64_t tb = t0 + (int64_t)own1 * kChunk < t1 ? t0 + (int64_t)own1 * kChunk : t1;
      for (int64_t idx = tid; idx < (tb - ta) * kVs; idx += kPassThreads)
        a.o[((ta + idx / kVs) * HV + h) * V + v0 + idx % kVs] = 0;
      continue;
    }
    if (own0 >= own1) continue;  // no chunk of this sequence in this part
    const int slot = a.state_idx[n];
    float* st = a.pool + ((size_t)slot * HV + h) * V * K;
    const size_t rec_stride = (size_t)HV * kRecBytes;
    scol = true;
    auto store_state = [&](float* dst) {  // S into a [V][K] FP32 state
      if (scol) {
        float4* d = reinterpret_cast<float4*>(dst + (size_t)(v0 + jc) * K + cc0);
        d[0] = make_float4(S[0], S[1], S[2], S[3]);
        d[1] = make_float4(S[4], S[5], S[6], S[7]);
      } else {
#pragma unroll
        for (int jj = 0; jj < kColsPerThread; ++jj) dst[(size_t)(v0 + j0 + jj) * K + c] = S[jj];
      }
    };
    // Everything below reads the chunk transform's records: with a dependent
    // launch, this is where the transform's completion is awaited (a no-op
    // after the first item).
    grid_dependency_wait();
    // A bound on the slice's states before they are computed: with
    // L2-normalised keys, beta = sigmoid(raw) < 1 and g <= 0, every map has norm
    // <= 1, so ||S_{c+1}|| <= ||S_c|| + ||B_c|| (the records keep ||B_c||).
    const bool bounded = a.gate.use_qk_l2norm && a.gate.beta_is_raw && (!a.gate.A_log || a.gate.lower_bound <= 0.f);
    const float* s_start = a.init_states ? a.init_states + ((size_t)n * HV + h) * V * K : st;  // the sequence's
    auto meta_of = [&](int j) -> float2 {  // {tau, ||B_c||} of the sequence's chunk j, this slice
      return __ldcg(reinterpret_cast<const float2*>(a.ws + ((size_t)(s_cbase + j) * HV + h) * kRecBytes +
                                                    kRecMeta) + slice);
    };
    if (bounded && warp < kPassEpiThreads / 32) {  // ||S_start[:, slice]||^2 by warp
      float sq = 0.f;
#pragma unroll
      for (int jj = 0; jj < kColsPerThread; ++jj) {
        const float x = s_start[(size_t)(v0 + j0 + jj) * K + row];
        sq += x * x;
      }
      sq = warp_sum(sq);
      if (lane == 0) s_pn[warp] = sq;
    }
    __syncthreads();
    // Part k > 0 starts at the latest chunk j + 1 <= own0 (j >= own0 - 32)
    // whose chain product is left out whatever S_j is -- an all-zero map, or
    // tau_j at least twice the bound on S_j -- so that S_{j+1} = B_j bit for
    // bit; else at the sequence's first chunk.  It runs the chunks before own0
    // again without writing their outputs.  Part 0 starts at own0 = 0.
    if (warp == 0) {
      float s0n = 0.f;
      if (bounded) {
        float t = 0.f;
        for (int w = 0; w < kPassEpiThreads / 32; ++w) t += s_pn[w];
        s0n = sqrtf(t) * kNormRoundUp;
      }
      int cs = 0;
      float bnd0 = s0n;  // bound on the run's start state
      if (own0 > 0) {
        float pre = 0.f;  // sum of ||B_c|| over c < own0: with s0n, a bound on every S_j, j <= own0
        if (bounded) {
          for (int j = lane; j < own0; j += 32) pre += meta_of(j).y;
          pre = warp_sum(pre);
        }
        const float bnd = (s0n + pre) * kNormRoundUp;
        const int j = own0 - 1 - lane;
        const float2 mj = j >= 0 ? meta_of(j) : make_float2(0.f, 0.f);
        const bool cut = j >= 0 && (__float_as_uint(mj.x) == 0x7f800000u || (bounded && 2.f * bnd <= mj.x));
        const uint32_t m = __ballot_sync(0xffffffffu, cut);
        if (m) {
          const int l = __ffs(m) - 1;
          cs = own0 - l;
          bnd0 = __shfl_sync(0xffffffffu, mj.y, l);  // S_cs = B_{cs-1}
        }
      }
      if (lane == 0) {
        s_cs = cs;
        s_bnd0 = bnd0;
      }
    }
    __syncthreads();
    const int cs = s_cs;
    const int nrun = own1 - cs;   // chunks run here, from chunk cs
    const int emit0 = own0 - cs;  // the first of them whose outputs are written
    const uint8_t* ws_head = a.ws + ((size_t)(s_cbase + cs) * HV + h) * kRecBytes;

    // Chunk ci's {tau, ||B_c||} for this slice (tau = +inf: M_c is all zero and
    // not stored), and the decisions every role takes the same way from them,
    // from the running bound on the chunk's start state (s_bnd0 plus the
    // ||B_c|| of the chunks before, added in order) and from the per-warp
    // maxima of that state.
    auto meta_at = [&](int ci) -> float2 {
      return __ldcg(reinterpret_cast<const float2*>(ws_head + (size_t)ci * rec_stride + kRecMeta) + slice);
    };
    auto map_stored = [](float tau) { return __float_as_uint(tau) != 0x7f800000u; };
    // left out whatever the state: the bound (doubled) is within tau
    auto certain_skip = [&](float tau, float bnd) { return bounded && 2.f * bnd <= tau; };
    // the M_c stage is copied and taken only for a product that may run
    auto m_needed = [&](float2 m, float bnd) { return map_stored(m.x) && !certain_skip(m.x, bnd); };
    auto state_max = [&](int b) -> float {  // max|S| of the state in buffer b (NaN is largest)
      uint32_t m = 0u;
#pragma unroll
      for (int w = 0; w < kPassEpiThreads / 32; ++w) m = max(m, s_pmax[b][w]);
      return __uint_as_float(m);
    };
    // The product is left out iff !m_needed, or else iff max|S| <= tau, where
    // max|S| comes from the per-warp maxima the epilogue publishes only then.

    if (copy_warp) {
      // ---- copy warp (one lane) ----
      if (lane == 0) {
        auto rec_of = [&](int cj) { return ws_head + (size_t)cj * rec_stride; };
        auto prefetch_record = [&](int cj, bool with_m) {  // the operand tiles, this slice of B_c and P Util
          const uint8_t* rec = rec_of(cj);
          if (with_m) tc::bulk_prefetch_l2(rec + kRecM, kStMBytes);
          tc::bulk_prefetch_l2(rec + kRecQ, kStQBytes);
          tc::bulk_prefetch_l2(rec + kRecB + slice * (kVs * kHeadDim * 4), kVs * kHeadDim * 4);
          tc::bulk_prefetch_l2(rec + kRecOi + slice * (kVs * kChunk * 4), kVs * kChunk * 4);
        };
        auto meta_ahead = [&](int cj) { return cj < nrun ? meta_at(cj) : make_float2(0.f, 0.f); };
        // chunks cj .. cj + 3, and the bound on chunk cj's start state
        float2 ta0 = meta_ahead(0), ta1 = meta_ahead(1), ta2 = meta_ahead(2), ta3 = meta_ahead(3);
        float bnd = s_bnd0;
        for (int cj = 1; cj < kPassL2Ahead && cj < nrun; ++cj)
          prefetch_record(cj, cj == 1 ? m_needed(ta1, bnd + ta0.y) : m_needed(ta2, (bnd + ta0.y) + ta1.y));
        int m_issued = s_m_issued, q_issued = s_q_issued;  // M_c and Q' copies issued by the CTA
        bool abort = false;
        for (int cj = 0; cj < nrun && !abort; ++cj) {
          const int gj = g0 + cj;  // the CTA's chunk
          if (m_needed(ta0, bnd)) {  // the M_c stage m_issued & 1 last held copy m_issued - 2
            if (m_issued >= 2 && !tc::mbar_wait(&m_free[m_issued & 1], ((m_issued - 2) >> 1) & 1)) {
              abort = true;
              break;
            }
            tc::fence_async_smem();
            issue_copy(smb + (m_issued & 1) * kStageBytes + kStM, rec_of(cj) + kRecM, kStMBytes, &m_full[m_issued & 1]);
            ++m_issued;
          }
          // the Q' stage gj & 1 held chunk gj - 2's Q': free once its output product is done
          if (gj >= 2 && !tc::mbar_wait(&o_bar[(gj - 2) % kOBufs], ((gj - 2) / kOBufs) & 1)) {
            abort = true;
            break;
          }
          tc::fence_async_smem();
          issue_copy(smb + (gj & 1) * kStageBytes + kStQ, rec_of(cj) + kRecQ, kStQBytes, &q_full[gj & 1]);
          ++q_issued;
          if (cj + kPassL2Ahead < nrun)
            prefetch_record(cj + kPassL2Ahead, m_needed(ta3, ((bnd + ta0.y) + ta1.y) + ta2.y));
          bnd = bnd + ta0.y;
          ta0 = ta1;
          ta1 = ta2;
          ta2 = ta3;
          ta3 = meta_ahead(cj + 4);
        }
        s_m_issued = m_issued;
        s_q_issued = q_issued;
        if (abort) {
          s_abort = 1;
          set_error(a.err_flag, KDA_DEVERR_TIMEOUT);
        }
      }
    } else if (mma_warp) {
      // ---- MMA warp (one lane) ----
      if (lane == 0) {
        auto issue_output = [&](int cj) {  // the CTA's chunk cj: output product (Q' stage cj & 1, state buffer cj % 3)
          const uint32_t qq = tc::smem_u32(smb + (cj & 1) * kStageBytes + kStQ);
          const uint32_t sb2 = tc::smem_u32(smb + kSmS + (cj % kSBufs) * kSmSBytes);
          const uint32_t dO = tmem + 64 + 64 * (cj % kOBufs);
#pragma unroll
          for (int k = 0; k < 8; ++k) {  // Q' [S_hi | S_lo]; Q' atom columns are 64 rows (8 KB) apart
            const uint32_t koff = (k & 3) * 32;
            tc::mma_bf16(dO, tc::sw128_desc(qq + (k >> 2) * (kChunk * 128) + koff),
                         tc::sw128_desc(sb2 + (k >> 2) * (2 * kVs * 128) + koff), idescO, k > 0);
          }
          tc::mma_commit(&o_bar[cj % kOBufs]);
        };
        float2 meta = meta_at(0);
        float bnd = s_bnd0;       // bound on chunk ci's start state
        int m_used = s_m_used;    // M_c stages taken by the CTA
        bool abort = false;
        for (int ci = 0; ci < nrun && !abort; ++ci) {
          const int gi = g0 + ci;  // the CTA's chunk
          {
            const float2 meta_next = ci + 1 < nrun ? meta_at(ci + 1) : make_float2(0.f, 0.f);
            const int b = gi % kSBufs;
            // state operand of chunk ci written (the item's first by the prologue)
            if (!tc::mbar_wait(&s_ready[b], (gi / kSBufs) & 1)) {
              abort = true;
              break;
            }
            // the state's maximum is published (and read) only where it decides
            const bool skip = !m_needed(meta, bnd) || state_max(b) <= meta.x;
            if (m_needed(meta, bnd)) {
              if (!tc::mbar_wait(&m_full[m_used & 1], (m_used >> 1) & 1)) {
                abort = true;
                break;
              }
              if (!skip) {
                tc::tc_fence_after();
                const uint32_t mh = tc::smem_u32(smb + (m_used & 1) * kStageBytes + kStM), ml = mh + 128 * 128 * 2;
                const uint32_t sb2 = tc::smem_u32(smb + kSmS + b * kSmSBytes);
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // M_hi [S_hi | S_lo]
                  const uint32_t koff = (k & 3) * 32;
                  tc::mma_bf16(dch, tc::sw128_desc(mh + (k >> 2) * (128 * 128) + koff),
                               tc::sw128_desc(sb2 + (k >> 2) * (2 * kVs * 128) + koff), idesc2, k > 0);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // + M_lo S_hi, into the S_lo half
                  const uint32_t koff = (k & 3) * 32;
                  tc::mma_bf16(dch + kVs, tc::sw128_desc(ml + (k >> 2) * (128 * 128) + koff),
                               tc::sw128_desc(sb2 + (k >> 2) * (2 * kVs * 128) + koff), idesc1, true);
                }
                tc::mma_commit(&ch_bar);
                tc::mma_commit(&m_free[m_used & 1]);
              } else {
                mbar_arrive(&m_free[m_used & 1]);  // landed and not read
              }
              ++m_used;
            }
            bnd = bnd + meta.y;
            meta = meta_next;
          }
          // chunk ci's output product, behind its chain product
          if (!tc::mbar_wait(&q_full[gi & 1], (gi >> 1) & 1)) {
            abort = true;
            break;
          }
          tc::tc_fence_after();
          issue_output(gi);
        }
        s_m_used = m_used;
        if (abort) {
          s_abort = 1;
          set_error(a.err_flag, KDA_DEVERR_TIMEOUT);
        }
      }
    } else {
      // ---- epilogue warps ----
      auto load_b = [&](int ci, bool col, float (&b)[kColsPerThread]) {  // B_c, [slice][column][channel]
        const float* src = reinterpret_cast<const float*>(ws_head + (int64_t)ci * (int64_t)rec_stride + kRecB) +
                           slice * kVs * kHeadDim;
        if (col) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(src + jc * kHeadDim + cc0));
          const float4 y = __ldcg(reinterpret_cast<const float4*>(src + jc * kHeadDim + cc0) + 1);
          b[0] = x.x; b[1] = x.y; b[2] = x.z; b[3] = x.w;
          b[4] = y.x; b[5] = y.y; b[6] = y.z; b[7] = y.w;
        } else {
#pragma unroll
          for (int jj = 0; jj < kColsPerThread; ++jj) b[jj] = __ldcg(src + (j0 + jj) * kHeadDim + c);
        }
      };
      auto load_pu = [&](int ci, float4& u0, float4& u1) {  // P Util rows t, [slice][quad][64][4]
        const float4* src = reinterpret_cast<const float4*>(ws_head + (size_t)ci * rec_stride + kRecOi) +
                            (slice * (kVs / 4) + j0 / 4) * kChunk + (quad * 16 + (lane & 15));
        u0 = __ldcg(src);
        u1 = __ldcg(src + kChunk);
      };
      if (cs == 0) {  // the sequence's start state (staged by the transform when run in parts)
        const float4* s0 = reinterpret_cast<const float4*>(s_start + (size_t)(v0 + jc) * K + cc0);
        const float4 x = s0[0], y = s0[1];
        S[0] = x.x; S[1] = x.y; S[2] = x.z; S[3] = x.w;
        S[4] = y.x; S[5] = y.y; S[6] = y.z; S[7] = y.w;
      } else {  // S_cs = B_{cs-1}: its product is left out whatever the state
        load_b(-1, true, S);
      }
      auto publish_max = [&](int buf) {  // this warp's max|S| for buffer buf's state
        uint32_t m = 0u;
#pragma unroll
        for (int jj = 0; jj < kColsPerThread; ++jj) m = max(m, __float_as_uint(S[jj]) & 0x7fffffffu);
#pragma unroll
        for (int o = 16; o; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) s_pmax[buf][warp] = m;
      };
      auto write_state_operand = [&](int buf) {  // rows j: S_hi[:, j]; rows 32 + j: S_lo[:, j]
        uint8_t* S2 = smb + kSmS + buf * kSmSBytes;
        if (scol) {
          uint4 hi, lo;
          split8(S, hi, lo);
          *reinterpret_cast<uint4*>(S2 + tc::sw128_offset(jc, cc0, 2 * kVs)) = hi;
          *reinterpret_cast<uint4*>(S2 + tc::sw128_offset(kVs + jc, cc0, 2 * kVs)) = lo;
        } else {
#pragma unroll
          for (int jj = 0; jj < kColsPerThread; ++jj) {
            uint16_t hi, lo;
            tc::split_bf16(S[jj], hi, lo);
            *reinterpret_cast<uint16_t*>(S2 + tc::sw128_offset(j0 + jj, c, 2 * kVs)) = hi;
            *reinterpret_cast<uint16_t*>(S2 + tc::sw128_offset(kVs + j0 + jj, c, 2 * kVs)) = lo;
          }
        }
      };
      auto write_intermediate = [&](int ci) {  // S is the start state of chunk ci
        if (!a.intermediate || ci < emit0) return;
        const int64_t cid = s_cbase + cs + ci;
        if (cid < a.inter_chunks) {
          store_state(a.intermediate + ((size_t)cid * HV + h) * V * K);
        } else if (tid == 0 && slice == 0) {
          set_error(a.err_flag, KDA_DEVERR_INTERMEDIATE);
        }
      };
      const uint32_t lane_addr = (static_cast<uint32_t>(quad * 32) << 16) + j0;
      // chunk cj's output: token 16 q + l is in TMEM lane 32 q + l (l < 16)
      const int orow = quad * 16 + (lane & 15);
      auto output = [&](int cj, const float4& u0, const float4& u1) -> bool {
        const int gj = g0 + cj;  // the CTA's chunk
        const bool ok = tc::mbar_wait(&o_bar[gj % kOBufs], (gj / kOBufs) & 1);
        tc::tc_fence_after();
        float dh[kColsPerThread], dl[kColsPerThread];
        const uint32_t dO = tmem + 64 + 64 * (gj % kOBufs);
        tc::tmem_ld8(dO + lane_addr, dh);
        tc::tmem_ld8(dO + lane_addr + kVs, dl);
        const float oo[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
        float x[8];
#pragma unroll
        for (int jj = 0; jj < kColsPerThread; ++jj) x[jj] = a.gate.scale * (dh[jj] + dl[jj] + oo[jj]);
        const int64_t tcj = t0 + (int64_t)(cs + cj) * kChunk;
        const int len = (int)(t1 - tcj < kChunk ? t1 - tcj : kChunk);
        if (lane < 16 && orow < len && cj >= emit0)
          *reinterpret_cast<uint4*>(a.o + ((tcj + orow) * HV + h) * V + v0 + j0) =
              make_uint4(pack_out16x2<F16>(x[0], x[1]), pack_out16x2<F16>(x[2], x[3]),
                         pack_out16x2<F16>(x[4], x[5]), pack_out16x2<F16>(x[6], x[7]));
        tc::tc_fence_before();
        return ok;
      };
      auto meta_ahead = [&](int ci) { return ci < nrun ? meta_at(ci) : make_float2(0.f, 0.f); };
      float4 pu0, pu1, pp0 = make_float4(0.f, 0.f, 0.f, 0.f), pp1 = pp0;  // pp: previous chunk's P Util
      float bb[kColsPerThread];                                         // the current chunk's B_c
      float2 meta = meta_at(0), meta1 = meta_ahead(1);  // the current and the next chunk's
      float bnd = s_bnd0;  // bound on the current chunk's start state
      bool bcol = !m_needed(meta, bnd);  // B_c (and then S) by column: the product is certainly left out
      load_b(0, bcol, bb);
      load_pu(0, pu0, pu1);
      // the buffer's last readers, the previous item's products, are done: this
      // warp waited for every one of its outputs
      const int b0 = g0 % kSBufs;
      publish_max(b0);
      write_state_operand(b0);
      write_intermediate(0);
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_ready[b0]);
      bool ok = tc::mbar_wait(&s_ready[b0], (g0 / kSBufs) & 1);
      float smax = state_max(b0);  // max|S| of the current chunk's start state
      for (int ci = 0; ci < nrun && ok; ++ci) {
        const bool more = ci + 1 < nrun;
        // the next chunk's B_c, P Util and the threshold after it, landing
        // while this one finishes
        const bool ncol = !m_needed(meta1, bnd + meta.y);
        float nbb[kColsPerThread];
        float4 nu0 = pu0, nu1 = pu1;
        float2 meta2 = make_float2(0.f, 0.f);
        if (more) {
          load_b(ci + 1, ncol, nbb);
          load_pu(ci + 1, nu0, nu1);
          meta2 = meta_ahead(ci + 2);
        }
        // S_{ci+1} = M_c S_ci + B_c, or B_c where the product cannot change it
        scol = bcol;
        if (m_needed(meta, bnd) && !(smax <= meta.x)) {
          if (!tc::mbar_wait(&ch_bar, nchain & 1)) ok = false;
          ++nchain;
          tc::tc_fence_after();
          float dh[kColsPerThread], dl[kColsPerThread];
          tc::tmem_ld8(dch + lane_addr, dh);
          tc::tmem_ld8(dch + lane_addr + kVs, dl);
#pragma unroll
          for (int jj = 0; jj < kColsPerThread; ++jj) S[jj] = dh[jj] + dl[jj] + bb[jj];
        } else {
#pragma unroll
          for (int jj = 0; jj < kColsPerThread; ++jj) S[jj] = bb[jj];
        }
        const int nb = (g0 + ci + 1) % kSBufs;
        // does chunk ci + 1's decision need the maximum of S_{ci+1}?
        const bool need_next = more && !ncol;
        if (more) {
          // its buffer's last readers, chunk ci - 2's products, finished before
          // chunk ci - 2's output product did, which this warp has waited for
          if (need_next) publish_max(nb);
          write_state_operand(nb);
          tc::fence_async_smem();
          tc::tc_fence_before();
          __syncwarp();  // the warp's operand writes (and TMEM reads) precede its arrival
          if (lane == 0) mbar_arrive(&s_ready[nb]);  // the MMA warp may issue chunk ci + 1
          write_intermediate(ci + 1);
        }
        if (ci >= 1 && !output(ci - 1, pp0, pp1)) ok = false;  // issued behind chunk ci's chain product
        if (need_next) {  // every epilogue warp's maximum of S_{ci+1}
          if (!tc::mbar_wait(&s_ready[nb], ((g0 + ci + 1) / kSBufs) & 1)) ok = false;
          smax = state_max(nb);
        }
        pp0 = pu0; pp1 = pu1;
        pu0 = nu0; pu1 = nu1;
        if (more) {
#pragma unroll
          for (int jj = 0; jj < kColsPerThread; ++jj) bb[jj] = nbb[jj];
        }
        bcol = ncol;
        bnd = bnd + meta.y;
        meta = meta1;
        meta1 = meta2;
      }
      if (ok && !output(nrun - 1, pp0, pp1)) ok = false;
      if (!ok) {
        s_abort = 1;
        set_error(a.err_flag, KDA_DEVERR_TIMEOUT);
      }
    }
    __syncthreads();
    if (!s_abort && !mma_warp && !copy_warp && part == parts - 1) store_state(st);
    g0 += nrun;
  }  // items
  if (copy_warp && lane == 0) {
    // no copy may outlive the CTA: the last two of each kind are the latest
    // phases of their barriers
    const int m_issued = s_m_issued, q_issued = s_q_issued;
    for (int j = m_issued - 2 > 0 ? m_issued - 2 : 0; j < m_issued; ++j)
      tc::mbar_wait(&m_full[j & 1], (j >> 1) & 1, 1u << 20);
    for (int j = q_issued - 2 > 0 ? q_issued - 2 : 0; j < q_issued; ++j)
      tc::mbar_wait(&q_full[j & 1], (j >> 1) & 1, 1u << 20);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// Given log-decays (A_log absent): the chunk transform's decay windows need
// every per-token log-decay in [kMinLogDecay, 0].  Each thread checks eight
// consecutive values of the real token rows (padding rows are never read); a
// value outside the range, or NaN, flags its sequence, which the transform and
// the state pass then skip and the token-by-token path computes.
template <bool F16>
__global__ void __launch_bounds__(256) decay_check_kernel(const PrefillArgs a, int32_t* flags) {
  const int64_t words_per_row = (int64_t)a.HV * kHeadDim / 8;
  const int64_t words = a.total_tokens * words_per_row;
  const uint4* g = reinterpret_cast<const uint4*>(a.g);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < words;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 w = __ldg(g + i);
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
    bool bad = false;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = in16_to_float<F16>((uint16_t)(u[e] & 0xffffu));
      const float hi = in16_to_float<F16>((uint16_t)(u[e] >> 16));
      bad |= !(lo >= kMinLogDecay && lo <= 0.f) || !(hi >= kMinLogDecay && hi <= 0.f);
    }
    if (bad) {
      const int64_t row = i / words_per_row;
      int n = 0;
      if (a.cu_seqlens) {  // last sequence whose start is <= row (binary search)
        int lo_n = 0, hi_n = a.num_seqs - 1;
        while (lo_n < hi_n) {
          const int mid = (lo_n + hi_n + 1) / 2;
          if ((int64_t)a.cu_seqlens[mid] <= row) lo_n = mid; else hi_n = mid - 1;
        }
        n = lo_n;
      } else {
        n = (int)(row / (a.total_tokens / a.num_seqs));
      }
      flags[n] = 1;
    }
  }
}

int64_t max_chunks(int num_seqs, int64_t total_tokens) {
  return total_tokens / kChunk + num_seqs;
}

// Workspace: the per-sequence flags of the given-decay check, then the
// (chunk, head) records, 256-byte aligned, then one start state per
// (sequence, head).
// per-sequence flags, then the multi-item pass's claim counter
size_t flags_bytes(int num_seqs) { return ((size_t)num_seqs * 4 + 4 + 255) & ~(size_t)255; }
constexpr size_t kStateBytes = (size_t)kHeadDim * kHeadDim * 4;

constexpr int kMaxDevices = 64;
bool g_attributes_set[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

// Sets the kernels' shared-memory limits and reads the SM count, once per
// device; returns the current device.
kda_status ensure_kernel_attributes(int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KDA_ERR_CUDA;
  *dev_out = dev;
  if (g_attributes_set[dev]) return KDA_OK;
  if (cudaFuncSetAttribute(chunk_transform_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kTransformTcSmem) != cudaSuccess ||
      cudaFuncSetAttribute(chunk_transform_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kTransformTcSmem) != cudaSuccess ||
      cudaFuncSetAttribute(state_pass_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kPassSmem) != cudaSuccess ||
      cudaFuncSetAttribute(state_pass_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kPassSmem) != cudaSuccess ||
      cudaFuncSetAttribute(state_pass_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kPassSmem) != cudaSuccess ||
      cudaFuncSetAttribute(state_pass_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)kPassSmem) != cudaSuccess ||
      cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return KDA_ERR_CUDA;
  g_attributes_set[dev] = true;
  return KDA_OK;
}

// Persistent transform: one CTA per SM (each holds a whole SM's shared
// memory), or one per unit when there are fewer units.
unsigned transform_grid(int64_t units, int dev) {
  return (unsigned)(units < g_num_sms[dev] ? units : g_num_sms[dev]);
}

cudaEvent_t g_stage_events[3] = {nullptr, nullptr, nullptr};

// The driver's tensor-map encoder, fetched once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<void*> fn{nullptr};
  void* f = fn.load(std::memory_order_relaxed);
  if (!f) {
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !f)
      return nullptr;
    fn.store(f, std::memory_order_relaxed);
  }
  return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
}

// Tensor map of a [T][heads][128] 16-bit tensor, box (box0 elements, 1 head,
// 64 tokens); elements outside the tensor land as zeros.
bool encode_rows(CUtensorMap* m, const void* base, int64_t heads, int64_t T, uint32_t box0) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dim[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)heads, (cuuint64_t)T};
  const cuuint64_t stride[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)heads * kHeadDim * 2};
  const cuuint32_t box[3] = {box0, 1u, (cuuint32_t)kChunk};
  const cuuint32_t estride[3] = {1u, 1u, 1u};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(base), dim, stride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Recorded as an external event node when the stream is being captured, so
// the event fires on every replay of the graph.
void record_stage(int i, cudaStream_t st) {
  if (g_stage_events[i]) cudaEventRecordWithFlags(g_stage_events[i], st, cudaEventRecordExternal);
}

}  // namespace kda

using namespace kda;

extern "C" size_t kda_prefill_workspace_size(kda_dims dims, int num_seqs, int64_t total_tokens) {
  if (num_seqs < 0 || total_tokens < 0 || dims.HV <= 0) return 0;
  // cu_seqlens are int32: larger calls are refused, and SIZE_MAX makes every
  // capacity check fail instead of wrapping
  if (total_tokens > INT32_MAX || dims.HV > (1 << 16)) return SIZE_MAX;
  return flags_bytes(num_seqs) + (size_t)max_chunks(num_seqs, total_tokens) * dims.HV * kRecBytes +
         (size_t)num_seqs * dims.HV * kStateBytes;
}

extern "C" kda_status kda_prefill(kda_dims dims, kda_gate gate, const kda_bf16* q,
                                  const kda_bf16* k, const kda_bf16* v, const kda_bf16* g,
                                  const kda_bf16* beta, int64_t gb_rows, float* state_pool,
                                  int pool_slots, const int32_t* state_idx,
                                  const int32_t* cu_seqlens, int num_seqs, int64_t total_tokens,
                                  kda_bf16* o, float* intermediate, int64_t intermediate_chunks,
                                  void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                  void* stream) {
  kda_status s = check_dims(dims);
  if (s != KDA_OK) return s;
  if (!state_pool || !state_idx) return KDA_ERR_NULL_ARG;  // indexed pool required
  if (num_seqs < 1 || total_tokens < 0 || pool_slots < 0) return KDA_ERR_SHAPE;
  if (total_tokens > INT32_MAX || (intermediate && intermediate_chunks < 0)) return KDA_ERR_SHAPE;
  if (gb_rows < total_tokens) return KDA_ERR_SHAPE;  // g/beta must cover every q token
  if (!cu_seqlens && total_tokens % num_seqs != 0) return KDA_ERR_SHAPE;
  if (total_tokens > 0 && (!q || !k || !v || !g || !beta || !o)) return KDA_ERR_NULL_ARG;
  PrefillArgs args{};
  s = check_gate(gate, &args.gate);
  if (s != KDA_OK) return s;
  // The chunk transform's decay-factor windows stay inside FP32 range for
  // per-token log-decays >= kMinLogDecay; a bounded gate that may go below it
  // takes the token-by-token path for every sequence.
  const bool token_path = gate.A_log && gate.lower_bound < kMinLogDecay;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g) || !aligned16(state_pool) ||
      !aligned16(o) || (intermediate && !aligned16(intermediate)))
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
  args.inter_chunks = intermediate ? intermediate_chunks : 0;
  args.ws = static_cast<uint8_t*>(workspace) + flags_bytes(num_seqs);
  args.err_flag = err_flag;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  // Kernel shared-memory limits are set once per device, on the first call
  // made with that device current.
  int dev = 0;
  if ((s = ensure_kernel_attributes(&dev)) != KDA_OK) return s;
  SeqPrefillArgs sp{};  // the token-by-token path's arguments
  sp.dims = dims;
  sp.gate = args.gate;
  sp.q = q;
  sp.k = k;
  sp.v = v;
  sp.g = g;
  sp.beta = beta;
  sp.pool = state_pool;
  sp.pool_slots = pool_slots;
  sp.state_idx = state_idx;
  sp.cu_seqlens = cu_seqlens;
  sp.num_seqs = num_seqs;
  sp.total_tokens = total_tokens;
  sp.o = o;
  sp.intermediate = intermediate;
  sp.inter_chunks = args.inter_chunks;
  sp.chunk_base = reinterpret_cast<int64_t*>(args.ws);  // the records' space, unused by then
  sp.err_flag = err_flag;
  if (token_path) {
    record_stage(0, st);
    s = launch_seq_prefill(sp, st);
    record_stage(1, st);
    record_stage(2, st);
    return s;
  }
  const int64_t chunks = max_chunks(num_seqs, total_tokens);
  uint8_t* const ws_states = args.ws + (size_t)chunks * dims.HV * kRecBytes;
  // the kernels for this call's 16-bit element type
  void (*const transform_kernel)(PrefillArgs, RowMaps) =
      dims.dtype == KDA_DTYPE_F16 ? chunk_transform_tc_kernel<true> : chunk_transform_tc_kernel<false>;
  record_stage(0, st);
  // Each (sequence, head, slice) chain in two parts where the grid still
  // fits the SMs, or, with more items than SMs anyway, where the sequences
  // average kMultiPartTokens tokens or more: the second part restarts behind
  // an all-zero map (see the pass), which halves the chain wherever the decay
  // is strong, and shorter items spread better over the CTAs.  The start
  // states are then staged by the transform.
  const int64_t items1 = (int64_t)kSlices * dims.HV * num_seqs;
  const int parts = total_tokens > 0 && (2 * items1 <= g_num_sms[dev] ||
                                         (items1 > g_num_sms[dev] && total_tokens >= (int64_t)num_seqs * kMultiPartTokens))
                        ? 2 : 1;
  // one CTA per (sequence, head, slice, part) item where they fit the SMs,
  // else as many CTAs as SMs, each claiming items from a counter
  const int64_t items = items1 * parts;
  const bool multi = items > g_num_sms[dev];
  args.item_counter = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(workspace) + (size_t)num_seqs * 4);
  if (!gate.A_log && total_tokens > 0) {
    // given log-decays: flag the sequences the chunk form cannot take (the
    // claim counter, right behind the flags, is cleared with them)
    int32_t* flags = static_cast<int32_t*>(workspace);
    if (cudaMemsetAsync(flags, 0, (size_t)num_seqs * 4 + (multi ? 4 : 0), st) != cudaSuccess) return KDA_ERR_CUDA;
    const int64_t words = total_tokens * dims.HV * kHeadDim / 8;
    const int64_t want = (words + 255) / 256;
    const unsigned blocks = (unsigned)(want < 8LL * g_num_sms[dev] ? want : 8LL * g_num_sms[dev]);
    (dims.dtype == KDA_DTYPE_F16 ? decay_check_kernel<true> : decay_check_kernel<false>)
        <<<blocks, 256, 0, st>>>(args, flags);
    if ((s = launch_status()) != KDA_OK) return s;
    args.seq_flags = flags;
  } else if (multi && cudaMemsetAsync(args.item_counter, 0, 4, st) != cudaSuccess) {
    return KDA_ERR_CUDA;
  }
  if (parts > 1) args.init_states = reinterpret_cast<float*>(ws_states);
  if (chunks > 0 && total_tokens > 0) {  // with no tokens every chunk is empty
    args.tx_units = chunks * dims.HV;
    RowMaps maps;
    if (!encode_rows(&maps.q, q, dims.H, total_tokens, kLdB) || !encode_rows(&maps.k, k, dims.H, total_tokens, kLdB) ||
        !encode_rows(&maps.v, v, dims.HV, total_tokens, kLdB) || !encode_rows(&maps.g, g, dims.HV, total_tokens, kHeadDim))
      return KDA_ERR_CUDA;
    transform_kernel<<<transform_grid(args.tx_units, dev), kTxThreads, kTransformTcSmem, st>>>(args, maps);
    if ((s = launch_status()) != KDA_OK) return s;
  }
  args.parts = parts;
  const dim3 grid((unsigned)(multi ? g_num_sms[dev] : (items > 0 ? items : 1)));
  const bool f16 = dims.dtype == KDA_DTYPE_F16;
  void (*const pass_kernel)(PrefillArgs) = multi ? (f16 ? state_pass_kernel<true, true> : state_pass_kernel<false, true>)
                                                 : (f16 ? state_pass_kernel<true, false> : state_pass_kernel<false, false>);
  if (g_stage_events[1]) {  // a stage event between the kernels: an ordinary launch
    record_stage(1, st);
    pass_kernel<<<grid, kPassThreads, kPassSmem, st>>>(args);
    s = launch_status();
  } else {  // dependent launch: the pass's CTAs start as the transform's leave
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kPassThreads);
    cfg.dynamicSmemBytes = kPassSmem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    s = cudaLaunchKernelEx(&cfg, pass_kernel, args) == cudaSuccess ? launch_status() : KDA_ERR_CUDA;
  }
  if (s == KDA_OK && args.seq_flags) {  // given log-decays: the flagged sequences, token by token
    sp.seq_flags = args.seq_flags;
    s = launch_seq_prefill(sp, st);
  }
  record_stage(2, st);
  return s;
}

extern "C" void kda_set_stage_events(void* const* events) {
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
