// Dense ancestor-mask export (tree training page, §Megatron 引擎: for
// compatibility with gradient checkpointing the Megatron engine passes a
// dense attention-mask tensor instead of a BlockMask object, because
// save_for_backward() serialises only tensors).
//
// M[b][i][j] = 1 iff key j is visible to query i of tree b, i.e. j is i or
// an ancestor of i: j <= i <= E[j] with E the subtree end of j's node
// (§树构建过程 mask caption); pad rows and pad columns are 0.  With the
// visible length len_j = E[j] - j + 1 (0 at pad keys, whose E is -1) the test
// is one unsigned compare: (unsigned)(i - j) < (unsigned)len_j.
//
// Layouts: TPA_MASK_U8 [B, T, T] bytes; TPA_MASK_BITS [B, T, T/32] uint32
// words, bit (j & 31) of word j >> 5.  `invert` writes the complement (1 =
// pair removed), the convention of boolean attention masks whose True entries
// block attention.
//
// The export is bound by HBM writes.  A CTA takes 128 query rows and a
// chunk of keys; each thread keeps its keys' E in registers (read once per
// CTA) and writes 16 bytes (U8: 16 keys) or 4 bytes (BITS: 32 keys) per row,
// the writes of a warp to one row being contiguous.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace {

constexpr int kThreadsDm = 256;
// Query rows per CTA (t_pad is a multiple of 128).  128 rows a CTA put the
// bit-packed export in one wave of CTAs: 2.2 -> 2.8 TB/s written on the
// GRPO-shaped trees with the row loop unrolled (2.9 -> 4.2 on the 56K-token tree).
constexpr int kRowsU8 = 128, kRowsBits = 128;

__global__ void __launch_bounds__(kThreadsDm) dense_mask_u8_kernel(const int32_t* __restrict__ subtree_end,
                                                                  int32_t t_pad, uint8_t* __restrict__ out,
                                                                  uint32_t invert) {
  const int b = blockIdx.z;
  const int j0 = (blockIdx.x * kThreadsDm + threadIdx.x) * 16;
  if (j0 >= t_pad) return;
  const int32_t* e = subtree_end + int64_t(b) * t_pad + j0;
  uint32_t len[16];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int4 v = reinterpret_cast<const int4*>(e)[q];
    const int ev[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = j0 + 4 * q + c;
      len[4 * q + c] = ev[c] >= j ? uint32_t(ev[c] - j + 1) : 0u;
    }
  }
  const uint32_t inv = invert ? 0x01010101u : 0u;
  uint8_t* dst = out + (int64_t(b) * t_pad + int64_t(blockIdx.y) * kRowsU8) * t_pad + j0;
  // four rows' 16-byte stores in flight per thread: 4.3 -> 6.7 TB/s written on
  // the GRPO-shaped trees (7.2 TB/s on the 56K-token tree)
#pragma unroll 4
  for (int r = 0; r < kRowsU8; ++r) {
    const int i = blockIdx.y * kRowsU8 + r;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t x = 0;
#pragma unroll
      for (int c = 0; c < 4; ++c) x |= uint32_t(uint32_t(i - (j0 + 4 * q + c)) < len[4 * q + c]) << (8 * c);
      w[q] = x ^ inv;
    }
    *reinterpret_cast<uint4*>(dst + int64_t(r) * t_pad) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// Bit-packed form.  For query row i, the 32 keys j0 + c of a thread's word
// are visible iff c <= i - j0 (a prefix of the word, one shift) and
// E[j0 + c] >= i.  Over a CTA's rows [i0, i1] the second set only shrinks:
// keys with E >= i1 stay in it, keys with E < i0 are never in it, and the
// others leave it after row E.  Keys of one compressed node share their E,
// so they leave in a few groups: the thread keeps the running set `cur` and
// peels off the group with the next-smallest E when that row is passed (a
// 32-key scan per group, once per CTA), instead of 32 compares per word.
__global__ void __launch_bounds__(kThreadsDm) dense_mask_bits_kernel(const int32_t* __restrict__ subtree_end,
                                                                    int32_t t_pad, uint32_t* __restrict__ out,
                                                                    uint32_t invert) {
  const int b = blockIdx.z;
  const int word = blockIdx.x * kThreadsDm + threadIdx.x;
  const int j0 = word * 32;
  if (j0 >= t_pad) return;
  const int32_t* e = subtree_end + int64_t(b) * t_pad + j0;
  int ev[32];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int4 v = reinterpret_cast<const int4*>(e)[q];
    ev[4 * q] = v.x, ev[4 * q + 1] = v.y, ev[4 * q + 2] = v.z, ev[4 * q + 3] = v.w;
  }
  const int i0 = blockIdx.y * kRowsBits, i1 = i0 + kRowsBits - 1;
  uint32_t always = 0u, dying = 0u;
#pragma unroll
  for (int c = 0; c < 32; ++c) {  // a pad key has E = -1 and is in neither set
    if (ev[c] >= i1) always |= 1u << c;
    else if (ev[c] >= i0) dying |= 1u << c;
  }
  uint32_t cur = always | dying;
  // the group of dying keys with the smallest E (e_next = INT_MAX when none)
  int e_next = 0x7fffffff;
  uint32_t g_next = 0u;
  auto next_group = [&]() {
    e_next = 0x7fffffff;
    g_next = 0u;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      if ((dying >> c) & 1u) {
        if (ev[c] < e_next) {
          e_next = ev[c];
          g_next = 1u << c;
        } else if (ev[c] == e_next) {
          g_next |= 1u << c;
        }
      }
    }
  };
  next_group();
  const uint32_t inv = invert ? 0xffffffffu : 0u;
  const int words = t_pad / 32;
  uint32_t* dst = out + (int64_t(b) * t_pad + int64_t(i0)) * words + word;
#pragma unroll 4
  for (int r = 0; r < kRowsBits; ++r) {
    const int i = i0 + r;
    const int d = i - j0;  // keys j0 .. j0 + d are at or before row i
    const uint32_t pre = d < 0 ? 0u : (d >= 31 ? 0xffffffffu : (2u << d) - 1u);
    dst[int64_t(r) * words] = (pre & cur) ^ inv;
    while (e_next == i) {  // these keys are seen by no row after i
      cur &= ~g_next;
      dying &= ~g_next;
      next_group();
    }
  }
}

}  // namespace

extern "C" uint64_t tpa_dense_mask_bytes(int32_t n_trees, int32_t t_pad, int32_t format) {
  if (n_trees < 1 || t_pad < 1 || t_pad % TPA_BLOCK_SIZE != 0) return 0;
  const uint64_t cells = uint64_t(n_trees) * uint64_t(t_pad) * uint64_t(t_pad);
  if (format == TPA_MASK_U8) return cells;
  if (format == TPA_MASK_BITS) return cells / 8;
  return 0;
}

extern "C" int tpa_dense_mask(const tpa_tree_view* tree, void* out, uint64_t out_bytes, int32_t format,
                              int32_t invert, void* stream) {
  TPA_NVTX_RANGE("tpa_dense_mask");
  if (!tree || !out || !tree->subtree_end || tree->n_trees < 1 || tree->n_trees > 65535 || tree->t_pad < 1 ||
      tree->t_pad % TPA_BLOCK_SIZE != 0)
    return TPA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(out) & 15) return TPA_ERR_INVALID_ARG;
  const uint64_t need = tpa_dense_mask_bytes(tree->n_trees, tree->t_pad, format);
  if (need == 0) return TPA_ERR_INVALID_ARG;
  if (out_bytes < need) return TPA_ERR_BUFFER_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int t = tree->t_pad;
  const uint32_t inv = invert ? 1u : 0u;
  if (format == TPA_MASK_U8) {
    const dim3 grid((t / 16 + kThreadsDm - 1) / kThreadsDm, t / kRowsU8, tree->n_trees);
    dense_mask_u8_kernel<<<grid, kThreadsDm, 0, st>>>(tree->subtree_end, t, static_cast<uint8_t*>(out), inv);
  } else {
    const dim3 grid((t / 32 + kThreadsDm - 1) / kThreadsDm, t / kRowsBits, tree->n_trees);
    dense_mask_bits_kernel<<<grid, kThreadsDm, 0, st>>>(tree->subtree_end, t, static_cast<uint32_t*>(out), inv);
  }
  TPA_CUDA_TRY(cudaGetLastError());
  return TPA_OK;
}
