// libtpa runtime glue: status strings, device check, metadata upload,
// block-mask buffer slicing and the status query that gathers every
// kernel's device status word.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "tpa.h"

namespace {
inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

struct MaskLayout {
  uint64_t cls, q_ptr, q_idx, k_ptr, k_idx, qmask, sched, line_count, total;
};

bool mask_layout(int32_t n_trees, int32_t t_pad, MaskLayout* L) {
  if (n_trees < 1 || t_pad < TPA_BLOCK_SIZE || t_pad % TPA_BLOCK_SIZE) return false;
  const uint64_t B = uint64_t(n_trees), n = uint64_t(t_pad / TPA_BLOCK_SIZE);
  const uint64_t cap = n * (n + 1) / 2;
  uint64_t o = 0;
  L->cls = o;   o = align256(o + B * n * n);
  L->q_ptr = o; o = align256(o + 4 * B * (n + 1));
  L->q_idx = o; o = align256(o + 4 * B * cap);
  L->k_ptr = o; o = align256(o + 4 * B * (n + 1));
  L->k_idx = o; o = align256(o + 4 * B * cap);
  L->qmask = o; o = align256(o + 2048 * B * cap);
  L->sched = o; o = align256(o + 4 * 16);
  L->line_count = o; o = align256(o + 4 * B * 2 * n);
  L->total = o;
  return true;
}
}  // namespace

extern "C" {

const char* tpa_status_string(int s) {
  switch (s) {
    case TPA_OK: return "TPA_OK";
    case TPA_ERR_INVALID_ARG: return "TPA_ERR_INVALID_ARG";
    case TPA_ERR_EMPTY_SEQUENCE: return "TPA_ERR_EMPTY_SEQUENCE";
    case TPA_ERR_SEQ_TOO_LONG: return "TPA_ERR_SEQ_TOO_LONG";
    case TPA_ERR_NO_MEMORY: return "TPA_ERR_NO_MEMORY";
    case TPA_ERR_CUDA: return "TPA_ERR_CUDA";
    case TPA_ERR_DEVICE_TIMEOUT: return "TPA_ERR_DEVICE_TIMEOUT";
    case TPA_ERR_UNSUPPORTED_DEVICE: return "TPA_ERR_UNSUPPORTED_DEVICE";
    case TPA_ERR_BUFFER_TOO_SMALL: return "TPA_ERR_BUFFER_TOO_SMALL";
    default: return "TPA_ERR_UNKNOWN";
  }
}

int tpa_version(void) { return 100; }

int tpa_device_check(void) {
  int dev = 0;
  cudaDeviceProp prop;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return TPA_ERR_CUDA;
  }
  return (prop.major == 10 && prop.minor == 3) ? TPA_OK : TPA_ERR_UNSUPPORTED_DEVICE;
}

int tpa_tree_upload(const tpa_tree* tree, void* dev_blob, uint64_t dev_bytes, void* stream) {
  TPA_NVTX_RANGE("tpa_tree_upload");
  if (!tree || !dev_blob || (reinterpret_cast<uintptr_t>(dev_blob) & 255)) return TPA_ERR_INVALID_ARG;
  const uint64_t need = tpa_internal_blob_bytes(tree);
  if (dev_bytes < need) return TPA_ERR_BUFFER_TOO_SMALL;
  TPA_CUDA_TRY(cudaMemcpyAsync(dev_blob, tpa_tree_host_blob(tree), need, cudaMemcpyHostToDevice,
                               static_cast<cudaStream_t>(stream)));
  return TPA_OK;
}

uint64_t tpa_blockmask_bytes(int32_t n_trees, int32_t t_pad) {
  MaskLayout L;
  return mask_layout(n_trees, t_pad, &L) ? L.total : 0;
}

int tpa_blockmask_make_view(void* base, int32_t n_trees, int32_t t_pad, tpa_blockmask_view* v) {
  MaskLayout L;
  if (!base || !v || (reinterpret_cast<uintptr_t>(base) & 255) || !mask_layout(n_trees, t_pad, &L))
    return TPA_ERR_INVALID_ARG;
  uint8_t* b = static_cast<uint8_t*>(base);
  const int32_t n = t_pad / TPA_BLOCK_SIZE;
  v->n_trees = n_trees;
  v->n_blk = n;
  v->cap = n * (n + 1) / 2;
  v->pad_ = 0;
  v->cls = b + L.cls;
  v->q_ptr = reinterpret_cast<int32_t*>(b + L.q_ptr);
  v->q_idx = reinterpret_cast<int32_t*>(b + L.q_idx);
  v->k_ptr = reinterpret_cast<int32_t*>(b + L.k_ptr);
  v->k_idx = reinterpret_cast<int32_t*>(b + L.k_idx);
  v->qmask = reinterpret_cast<uint32_t*>(b + L.qmask);
  v->sched = reinterpret_cast<uint32_t*>(b + L.sched);
  v->line_count = reinterpret_cast<int32_t*>(b + L.line_count);
  return TPA_OK;
}

int tpa_sync_status(void* stream) {
  TPA_NVTX_RANGE("tpa_sync_status");
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return TPA_ERR_CUDA;
  }
  int worst = TPA_OK;
  const int s[5] = {tpa_internal_status_classify(true), tpa_internal_status_logprobs(true),
                    tpa_internal_status_fwd(true), tpa_internal_status_bwd(true),
                    tpa_internal_status_lmh(true)};
  for (int x : s) {
    if (x == TPA_ERR_CUDA) return TPA_ERR_CUDA;
    if (x != TPA_OK) worst = x;
  }
  return worst;
}

}  // extern "C"
