// Declarations shared by the translation units of libtpa (not part of the ABI).
#pragma once
#include <cstdint>

#include "tpa.h"

// NVTX range around a library call, named after it, so that a timeline
// profiler shows where each call starts and ends on the host (header-only
// NVTX v3; without a profiler attached it costs a load and a branch).  Host
// builds without the CUDA headers get no ranges.
#if __has_include(<nvtx3/nvToolsExt.h>)
#include <nvtx3/nvToolsExt.h>
struct TpaNvtxRange {
  explicit TpaNvtxRange(const char* name) { nvtxRangePushA(name); }
  ~TpaNvtxRange() { nvtxRangePop(); }
  TpaNvtxRange(const TpaNvtxRange&) = delete;
  TpaNvtxRange& operator=(const TpaNvtxRange&) = delete;
};
#define TPA_NVTX_RANGE(name) TpaNvtxRange tpa_nvtx_range_(name)
#else
#define TPA_NVTX_RANGE(name) ((void)0)
#endif

uint64_t tpa_internal_blob_bytes(const tpa_tree* tree);

// Each CUDA translation unit keeps its own device status word; these read
// (and clear) it.  They return TPA_OK, TPA_ERR_DEVICE_TIMEOUT, TPA_ERR_INVALID_ARG
// (an input outside its range was skipped) or TPA_ERR_CUDA.
int tpa_internal_status_classify(bool clear);
int tpa_internal_status_logprobs(bool clear);
int tpa_internal_status_fwd(bool clear);
int tpa_internal_status_bwd(bool clear);
int tpa_internal_status_lmh(bool clear);

// The per-sequence gather of the log-prob pass (logprobs.cu), shared with
// the fused LM-head path: seq_entropy[t] = pos_entropy[position of token t],
// seq_logp[t] = pos_logp[position of token t+1] (0 at a sequence's end).
int tpa_internal_seq_gather(const tpa_tree_view* tree, const float* pos_logp, const float* pos_entropy,
                            float* seq_logp, float* seq_entropy, void* stream);
