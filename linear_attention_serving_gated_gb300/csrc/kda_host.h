// kda_host.h -- host-side argument checks shared by the entry points.
//
// The checks mirror the ValueErrors of the pages' contracts: a missing pool
// or index array (chunk_kda: "KDA prefill requires an indexed initial-state
// pool"), gate/beta rows that do not cover every q token, non-power-of-two K
// or V and a gate input whose width is not HV*K (validate_packed_decode_inputs)
// -- all from "PR #35197 report: fix(kernel) Fix Helion small-token prefill
// bug", key source snippets of kda_prefill.py and kda_decode.py.
#pragma once

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/kda.h"
#include "kda_device.cuh"

namespace kda {

inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline kda_status check_dims(const kda_dims& d) {
  if (d.H <= 0 || d.HV <= 0 || d.K <= 0 || d.V <= 0) return KDA_ERR_SHAPE;
  if (!is_pow2(d.K) || !is_pow2(d.V)) return KDA_ERR_UNSUPPORTED;
  // grouped value heads: HV a multiple of H, value head h reading q/k head h / (HV / H)
  if (d.HV % d.H != 0 || d.K != kHeadDim || d.V != kHeadDim) return KDA_ERR_UNSUPPORTED;
  if (d.dtype != KDA_DTYPE_BF16 && d.dtype != KDA_DTYPE_F16) return KDA_ERR_UNSUPPORTED;
  return KDA_OK;
}

inline kda_status check_gate(const kda_gate& g, GateArgs* out) {
  if (g.A_log && isnan(g.lower_bound)) return KDA_ERR_UNSUPPORTED;  // unbounded gate
  if (g.dt_bias && !aligned16(g.dt_bias)) return KDA_ERR_ALIGNMENT;
  out->A_log = g.A_log;
  out->dt_bias = g.A_log ? g.dt_bias : nullptr;
  out->lower_bound = g.lower_bound;
  out->beta_is_raw = g.beta_is_raw;
  out->use_qk_l2norm = g.use_qk_l2norm;
  out->scale = g.scale;
  return KDA_OK;
}

inline kda_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// Profiling aid: records stage event i (see kda_set_stage_events) on the
// stream if one is set.
void record_stage(int i, cudaStream_t st);

// The prefill's token-by-token path, for sequences whose log-decays the
// chunk form's decay windows cannot take: one step per token like decode, the
// state in registers, o and chunk-start states written per token and chunk,
// the final state once.  seq_flags non-null: only the flagged sequences run.
// chunk_base: device scratch of num_seqs int64 (written when intermediate is
// set), stream-ordered after every earlier use of that memory.
struct SeqPrefillArgs {
  kda_dims dims;
  GateArgs gate;
  const kda_bf16 *q, *k, *v, *g, *beta;
  float* pool;
  int pool_slots;
  const int32_t* state_idx;
  const int32_t* cu_seqlens;
  int num_seqs;
  int64_t total_tokens;
  const int32_t* seq_flags;
  kda_bf16* o;
  float* intermediate;
  int64_t inter_chunks;
  int64_t* chunk_base;
  int32_t* err_flag;
};
kda_status launch_seq_prefill(const SeqPrefillArgs& p, cudaStream_t stream);

}  // namespace kda
