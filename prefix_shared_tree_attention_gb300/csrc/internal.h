// Declarations shared by the translation units of libtpa (not part of the ABI).
#pragma once
#include <cstdint>

#include "tpa.h"

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
