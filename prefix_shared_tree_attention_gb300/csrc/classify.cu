// Block classification of the packed trees (tree training page, §树构建过程
// step 4 "mask generation" and §注意力机制: a block mask with BLOCK_SIZE 128
// lets the attention skip empty blocks).
//
// Key j (real, j < n) is visible to query i iff j <= i <= E[j], E = subtree
// end of j's node.  For a tile (qb, kb) the number of visible pairs is
//   cnt = sum_{j in kb} max(0, min(E[j], q1) - max(j, q0) + 1),
// q0 = 128 qb, q1 = q0 + 127; the tile is EMPTY when cnt = 0, FULL when
// cnt = 128 * 128 and PARTIAL otherwise.  Two CSR lists follow: per query
// block its non-empty key blocks (forward), per key block its non-empty
// query blocks (backward), each entry 2 * block + (FULL ? 1 : 0), built by a
// count pass and a fill pass with one warp per line.  A third
// kernel writes, for every PARTIAL entry of the per-query-block list, the
// 128x128 visibility bits the forward applies (one 16-byte row per query).
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace {

__device__ unsigned int g_status_classify = 0;

constexpr int kB = TPA_BLOCK_SIZE;

// grid (n_blk, B), 128 threads: one CTA per key block; warp w handles query
// blocks qb = kb + w, kb + w + 4, ... with lane l covering keys l, l+32, ...
__global__ void __launch_bounds__(128) classify_kernel(const int32_t* __restrict__ subtree_end,
                                                        const int32_t* __restrict__ n_tokens,
                                                        int32_t t_pad, int32_t n_blk,
                                                        uint8_t* __restrict__ cls) {
  __shared__ int e_s[kB];
  __shared__ int emax_s[4];
  const int b = blockIdx.y, kb = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n = n_tokens[b];
  const int j = kb * kB + tid;
  const int e = (j < n) ? subtree_end[int64_t(b) * t_pad + j] : -1;
  e_s[tid] = e;
  int m = e;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) emax_s[warp] = m;
  __syncthreads();
  const int emax = max(max(emax_s[0], emax_s[1]), max(emax_s[2], emax_s[3]));
  uint8_t* out = cls + int64_t(b) * n_blk * n_blk + kb;   // column kb, row stride n_blk
  const int qb_last = (emax < 0) ? -1 : emax / kB;        // no key of this block reaches beyond
  for (int qb = warp; qb < n_blk; qb += 4) {
    int c = TPA_BLOCK_EMPTY;
    if (qb >= kb && qb <= qb_last) {
      const int q0 = qb * kB, q1 = q0 + kB - 1;
      int cnt = 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int jj = kb * kB + lane + 32 * u;
        const int ee = e_s[lane + 32 * u];
        if (ee >= 0) cnt += max(0, min(ee, q1) - max(jj, q0) + 1);
      }
      cnt = warp_sum(cnt);
      c = (cnt == 0) ? TPA_BLOCK_EMPTY : (cnt == kB * kB ? TPA_BLOCK_FULL : TPA_BLOCK_PARTIAL);
    }
    if (lane == 0) out[int64_t(qb) * n_blk] = uint8_t(c);
  }
}

// The two CSR lists, one warp per line (direction 0: the row of a query
// block, its non-empty key blocks; direction 1: the column of a key block,
// its non-empty query blocks).  csr_count_kernel counts each line's
// non-empty tiles; csr_fill_kernel takes a line's offset as the sum of the
// counts before it, and writes its entries in ascending order, 32 at a time
// with a ballot.  grid (ceil(n_blk / 8), B, 2), 256 threads: warp w of CTA x
// handles line 8x + w.
constexpr int kLinesPerCta = 8;

__device__ __forceinline__ uint8_t tile_of(const uint8_t* c, int n_blk, int dir, int line, int o) {
  return dir == 0 ? c[int64_t(line) * n_blk + o] : c[int64_t(o) * n_blk + line];
}

__global__ void __launch_bounds__(256) csr_count_kernel(const uint8_t* __restrict__ cls, int32_t n_blk,
                                                         int32_t* __restrict__ line_count) {
  const int b = blockIdx.y, dir = blockIdx.z;
  const int lane = threadIdx.x & 31;
  const int line = blockIdx.x * kLinesPerCta + (threadIdx.x >> 5);
  if (line >= n_blk) return;
  const uint8_t* c = cls + int64_t(b) * n_blk * n_blk;
  int cnt = 0;
  for (int o = lane; o < n_blk; o += 32) cnt += tile_of(c, n_blk, dir, line, o) != TPA_BLOCK_EMPTY;
  cnt = warp_sum(cnt);
  if (lane == 0) line_count[(int64_t(b) * 2 + dir) * n_blk + line] = cnt;
}

__global__ void __launch_bounds__(256) csr_fill_kernel(const uint8_t* __restrict__ cls, int32_t n_blk,
                                                        int32_t cap, const int32_t* __restrict__ line_count,
                                                        int32_t* __restrict__ q_ptr, int32_t* __restrict__ q_idx,
                                                        int32_t* __restrict__ k_ptr, int32_t* __restrict__ k_idx,
                                                        uint32_t* __restrict__ sched) {
  __shared__ int part_s[8];
  const int b = blockIdx.y, dir = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int line0 = blockIdx.x * kLinesPerCta;
  const int32_t* cnt = line_count + (int64_t(b) * 2 + dir) * n_blk;
  if (b == 0 && dir == 0 && blockIdx.x == 0 && tid < 16) sched[tid] = 0;  // work counters of the attention kernels
  // entries of the lines before this CTA's first one
  int part = 0;
  for (int i = tid; i < line0; i += blockDim.x) part += cnt[i];
  part = warp_sum(part);
  if (lane == 0) part_s[warp] = part;
  __syncthreads();
  int off = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) off += part_s[w];
  const int line = line0 + warp;
  if (line >= n_blk) return;
  for (int w = 0; w < warp; ++w) off += cnt[line0 + w];
  int32_t* ptr = (dir == 0 ? q_ptr : k_ptr) + int64_t(b) * (n_blk + 1);
  int32_t* idx = (dir == 0 ? q_idx : k_idx) + int64_t(b) * cap;
  if (lane == 0) {
    ptr[line] = off;
    if (line == n_blk - 1) ptr[n_blk] = off + cnt[line];
  }
  const uint8_t* c = cls + int64_t(b) * n_blk * n_blk;
  for (int o0 = 0; o0 < n_blk; o0 += 32) {
    const int o = o0 + lane;
    const uint8_t v = o < n_blk ? tile_of(c, n_blk, dir, line, o) : uint8_t(TPA_BLOCK_EMPTY);
    const unsigned mask = __ballot_sync(0xffffffffu, v != TPA_BLOCK_EMPTY);
    if (v != TPA_BLOCK_EMPTY) idx[off + __popc(mask & ((1u << lane) - 1u))] = 2 * o + (v == TPA_BLOCK_FULL ? 1 : 0);
    off += __popc(mask);
  }
}

// grid (n_blk, B), 128 threads: for every PARTIAL entry of query block qb's
// CSR row, thread r writes the 128-bit visibility row of query qb*128 + r:
// bit c of word c/32 is set iff key kb*128 + c is visible (j <= i <= E[j]).
__global__ void __launch_bounds__(128) qmask_kernel(const int32_t* __restrict__ subtree_end,
                                                     const int32_t* __restrict__ n_tokens, int32_t t_pad,
                                                     int32_t n_blk, int32_t cap,
                                                     const int32_t* __restrict__ q_ptr,
                                                     const int32_t* __restrict__ q_idx,
                                                     uint4* __restrict__ qmask) {
  __shared__ int e_s[kB];
  const int b = blockIdx.y, qb = blockIdx.x, r = threadIdx.x;
  const int n = n_tokens[b];
  const int i = qb * kB + r;
  const int32_t* ptr = q_ptr + int64_t(b) * (n_blk + 1);
  for (int e = ptr[qb]; e < ptr[qb + 1]; ++e) {
    const int ent = q_idx[int64_t(b) * cap + e];
    if (ent & 1) continue;  // FULL: no mask needed (uniform across the CTA)
    const int kb = ent >> 1;
    __syncthreads();
    const int jr = kb * kB + r;
    e_s[r] = (jr < n) ? subtree_end[int64_t(b) * t_pad + jr] : -1;
    __syncthreads();
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int c = 0; c < kB; ++c) {
      const int j = kb * kB + c;
      if (j <= i && i <= e_s[c]) w[c >> 5] |= 1u << (c & 31);
    }
    qmask[(int64_t(b) * cap + e) * kB + r] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

TPA_DEFINE_STATUS_READER(tpa_internal_status_classify, g_status_classify)

extern "C" int tpa_block_classify(const tpa_tree_view* tree, const tpa_blockmask_view* mask,
                                  void* stream) {
  TPA_NVTX_RANGE("tpa_block_classify");
  if (!tree || !mask || !tree->subtree_end || !tree->n_tokens || !mask->cls || !mask->q_ptr ||
      !mask->q_idx || !mask->k_ptr || !mask->k_idx || !mask->qmask || !mask->sched || !mask->line_count)
    return TPA_ERR_INVALID_ARG;
  if (tree->t_pad % kB || mask->n_blk != tree->t_pad / kB || mask->n_trees != tree->n_trees ||
      mask->n_blk > 1024 || tree->n_trees < 1)
    return TPA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int n_blk = mask->n_blk;
  classify_kernel<<<dim3(n_blk, tree->n_trees), 128, 0, st>>>(tree->subtree_end, tree->n_tokens,
                                                              tree->t_pad, n_blk, mask->cls);
  TPA_CUDA_TRY(cudaGetLastError());
  const dim3 lines((n_blk + kLinesPerCta - 1) / kLinesPerCta, tree->n_trees, 2);
  csr_count_kernel<<<lines, 256, 0, st>>>(mask->cls, n_blk, mask->line_count);
  TPA_CUDA_TRY(cudaGetLastError());
  csr_fill_kernel<<<lines, 256, 0, st>>>(mask->cls, n_blk, mask->cap, mask->line_count, mask->q_ptr, mask->q_idx,
                                         mask->k_ptr, mask->k_idx, mask->sched);
  TPA_CUDA_TRY(cudaGetLastError());
  qmask_kernel<<<dim3(n_blk, tree->n_trees), 128, 0, st>>>(tree->subtree_end, tree->n_tokens, tree->t_pad,
                                                           n_blk, mask->cap, mask->q_ptr, mask->q_idx,
                                                           reinterpret_cast<uint4*>(mask->qmask));
  TPA_CUDA_TRY(cudaGetLastError());
  return TPA_OK;
}
