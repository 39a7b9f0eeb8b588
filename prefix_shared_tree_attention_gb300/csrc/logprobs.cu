// Log-probabilities and entropies of a packed tree (tree training page,
// §对数概率计算): each tree row is processed exactly once (the node-level
// cache of the page), and the labels of that row — the next token inside its
// node and the first token of every child node — are gathered in the same
// pass; a second kernel regathers the per-position values per input sequence.
//
// Row kernel: one CTA streams one logits row (bf16, 16-byte vector loads)
// and keeps, per thread, the running max m, s = sum exp(x - m) and
// t = sum exp(x - m) * x; after a block reduction
//   lse = m + log s,   entropy = lse - t / s   (= -sum p log p),
//   pos_logp[c] = x[token c] - lse   for every child position c of the row.
// HBM-bound: each logits element is read once.
//
// A logit of -inf (a masked vocabulary entry) has p = 0 and adds nothing to
// s or t (p log p -> 0 as p -> 0); a row whose logits are all -inf has no
// distribution, and its entropy and log-probs come out NaN.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"

namespace {

__device__ unsigned int g_status_logprobs = 0;

constexpr int kRowThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

struct Acc {
  float m, s, t;  // running max, sum exp(x - m), sum exp(x - m) * x
};

__device__ __forceinline__ void acc_merge(Acc& a, const Acc& b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return;
  const float ca = ex2((a.m - m) * kLog2e), cb = ex2((b.m - m) * kLog2e);
  a.s = a.s * ca + b.s * cb;
  a.t = a.t * ca + b.t * cb;
  a.m = m;
}

// Masked entries: every bf16 value below -2^100 (-inf included; negative
// bf16 values grow as unsigned bits) is clamped to -2^100 (0xF180) before it
// is widened, with one unsigned 16x2 minimum per pair of values.  Next to any
// real logit its exponential is then exactly 0 and its t term 0 * x = 0, so
// it drops out of s and t as p log p -> 0 requires.  The clamp value is small
// enough that m * log2e and a whole row's sum of e * x stay finite while a
// thread has seen only masked entries (a row holds fewer than 2^27 entries).
// The row's label logits are read unclamped.
constexpr uint32_t kClampPair = 0xF180F180u;
constexpr float kMaskedMax = -1.0e30f;  // a row max at or below this: every entry was masked

__device__ __forceinline__ uint32_t clamp_neg_inf2(uint32_t w) {
  uint32_t r;
  asm("min.u16x2 %0, %1, %2;" : "=r"(r) : "r"(w), "r"(kClampPair));
  return r;
}

// Fold 8 values (one 16-byte vector) into the accumulator.
__device__ __forceinline__ void acc_add8(Acc& a, uint4 v) {
  v.x = clamp_neg_inf2(v.x);
  v.y = clamp_neg_inf2(v.y);
  v.z = clamp_neg_inf2(v.z);
  v.w = clamp_neg_inf2(v.w);
  float x[8] = {bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y),
                bf16_lo(v.z), bf16_hi(v.z), bf16_lo(v.w), bf16_hi(v.w)};
  float mc = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])),
                   fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
  if (mc > a.m) {
    const float c = ex2((a.m - mc) * kLog2e);
    a.s *= c;
    a.t *= c;
    a.m = mc;
  }
  const float mb = a.m * kLog2e;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float e = ex2(fmaf(x[i], kLog2e, -mb));
    a.s += e;
    a.t = fmaf(e, x[i], a.t);
  }
}

__device__ __forceinline__ void acc_add1(Acc& a, uint16_t raw) {
  const float x = bf16_lo(clamp_neg_inf2(raw));
  if (x > a.m) {
    const float c = ex2((a.m - x) * kLog2e);
    a.s *= c;
    a.t *= c;
    a.m = x;
  }
  const float e = ex2((x - a.m) * kLog2e);
  a.s += e;
  a.t = fmaf(e, x, a.t);
}

// grid (T_pad, B): CTA (p, b) handles tree position p of tree b.
__global__ void __launch_bounds__(kRowThreads) row_kernel(
    const uint16_t* __restrict__ logits, int64_t row_stride, int32_t layout, int32_t vocab,
    int32_t t_pad, int64_t total_rows, const int32_t* __restrict__ n_tokens,
    const int64_t* __restrict__ tok_base, const int32_t* __restrict__ tokens,
    const int32_t* __restrict__ parent, const int32_t* __restrict__ child_off,
    const int32_t* __restrict__ child_pos, float* __restrict__ pos_logp,
    float* __restrict__ pos_entropy) {
  const int p = blockIdx.x, b = blockIdx.y;
  const int64_t at = int64_t(b) * t_pad + p;
  const int n = n_tokens[b];
  if (!dbg_ok(n >= 0 && n <= t_pad, &g_status_logprobs)) return;
  if (p >= n) {  // padding position
    if (threadIdx.x == 0) {
      pos_logp[at] = 0.f;
      pos_entropy[at] = 0.f;
    }
    return;
  }
  const int64_t row = (layout == TPA_LOGITS_COMPACT) ? tok_base[b] + p : int64_t(b) * t_pad + p;
  if (layout == TPA_LOGITS_COMPACT && !dbg_ok(row >= 0 && row < total_rows, &g_status_logprobs)) return;
  const uint16_t* x = logits + row * row_stride;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int nvec = vocab >> 3;

  // Eight 16-byte loads in flight per thread, then four, then one: with 256
  // threads a row (eight CTAs an SM) this read 2.3 % faster than four loads
  // with 512 threads, and more loads or more threads a row were slower.
  Acc a{-INFINITY, 0.f, 0.f};
  int i = threadIdx.x;
  for (; i + 7 * kRowThreads < nvec; i += 8 * kRowThreads) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcs(xv + i + u * kRowThreads);
#pragma unroll
    for (int u = 0; u < 8; ++u) acc_add8(a, v[u]);
  }
  for (; i + 3 * kRowThreads < nvec; i += 4 * kRowThreads) {
    const uint4 v0 = __ldcs(xv + i);
    const uint4 v1 = __ldcs(xv + i + kRowThreads);
    const uint4 v2 = __ldcs(xv + i + 2 * kRowThreads);
    const uint4 v3 = __ldcs(xv + i + 3 * kRowThreads);
    acc_add8(a, v0);
    acc_add8(a, v1);
    acc_add8(a, v2);
    acc_add8(a, v3);
  }
  for (; i < nvec; i += kRowThreads) acc_add8(a, __ldcs(xv + i));
  for (int k = (nvec << 3) + threadIdx.x; k < vocab; k += kRowThreads)
    acc_add1(a, x[k]);

  // block reduction of (m, s, t)
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    Acc bo{__shfl_xor_sync(0xffffffffu, a.m, o), __shfl_xor_sync(0xffffffffu, a.s, o),
           __shfl_xor_sync(0xffffffffu, a.t, o)};
    acc_merge(a, bo);
  }
  __shared__ Acc part[kRowThreads / 32];
  __shared__ float lse_s;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) part[warp] = a;
  __syncthreads();
  if (warp == 0) {
    a = lane < kRowThreads / 32 ? part[lane] : Acc{-INFINITY, 0.f, 0.f};
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Acc bo{__shfl_xor_sync(0xffffffffu, a.m, o), __shfl_xor_sync(0xffffffffu, a.s, o),
             __shfl_xor_sync(0xffffffffu, a.t, o)};
      acc_merge(a, bo);
    }
    if (lane == 0) {
      // every entry -inf: no distribution, NaN entropy and log-probs
      const float lse = a.m > kMaskedMax ? a.m + __log2f(a.s) * kLn2 : __uint_as_float(0x7fc00000u);
      lse_s = lse;
      pos_entropy[at] = lse - a.t / a.s;
      if (parent[at] < 0) pos_logp[at] = 0.f;  // no parent row: no label for this position
    }
  }
  __syncthreads();
  const int c0 = child_off[int64_t(b) * (t_pad + 1) + p];
  const int c1 = child_off[int64_t(b) * (t_pad + 1) + p + 1];
  if (!dbg_ok(c0 >= 0 && c0 <= c1 && c1 <= t_pad, &g_status_logprobs)) return;
  for (int c = c0 + threadIdx.x; c < c1; c += kRowThreads) {
    const int cp = child_pos[int64_t(b) * t_pad + c];
    if (!dbg_ok(cp > p && cp < n, &g_status_logprobs)) continue;  // a child follows its parent
    const int tok = tokens[int64_t(b) * t_pad + cp];
    if (uint32_t(tok) < uint32_t(vocab)) {
      const float xl = __uint_as_float(uint32_t(x[tok]) << 16);
      pos_logp[int64_t(b) * t_pad + cp] = xl - lse_s;
    } else {  // a label outside the row: not read (the host refuses such trees)
      pos_logp[int64_t(b) * t_pad + cp] = __uint_as_float(0x7fc00000u);
      atomicOr(&g_status_logprobs, TPA_DEV_BAD_INPUT);
    }
  }
}

// grid (n_seqs): per input sequence s at token t,
//   seq_entropy[t] = pos_entropy[g_t],  seq_logp[t] = pos_logp[g_{t+1}] (0 at the end).
__global__ void __launch_bounds__(256) seq_gather_kernel(
    int32_t t_pad, int32_t n_trees, int64_t total_seq_tokens, const int32_t* __restrict__ n_tokens,
    const int32_t* __restrict__ seq_tree, const int64_t* __restrict__ seq_off,
    const int32_t* __restrict__ seq_pos, const float* __restrict__ pos_logp,
    const float* __restrict__ pos_entropy, float* __restrict__ seq_logp,
    float* __restrict__ seq_entropy) {
  const int s = blockIdx.x;
  const int64_t o0 = seq_off[s], o1 = seq_off[s + 1];
  const int tr = seq_tree[s];
  if (!dbg_ok(tr >= 0 && tr < n_trees && o0 >= 0 && o0 <= o1 && o1 <= total_seq_tokens, &g_status_logprobs))
    return;
  const int64_t base = int64_t(tr) * t_pad;
  const int n = TPA_DEBUG ? n_tokens[tr] : t_pad;
  for (int64_t i = o0 + threadIdx.x; i < o1; i += blockDim.x) {
    const int g0 = seq_pos[i], g1 = (i + 1 < o1) ? seq_pos[i + 1] : 0;
    if (!dbg_ok(g0 >= 0 && g0 < n && g1 >= 0 && g1 < n, &g_status_logprobs)) continue;
    seq_entropy[i] = pos_entropy[base + g0];
    seq_logp[i] = (i + 1 < o1) ? pos_logp[base + g1] : 0.f;
  }
}

}  // namespace

TPA_DEFINE_STATUS_READER(tpa_internal_status_logprobs, g_status_logprobs)

extern "C" int tpa_tree_logprobs_entropy(const tpa_tree_view* tree, const void* logits,
                                         int64_t row_stride, int32_t layout, int32_t vocab,
                                         float* pos_logp, float* pos_entropy, float* seq_logp,
                                         float* seq_entropy, void* stream) {
  TPA_NVTX_RANGE("tpa_tree_logprobs_entropy");
  if (!tree || !logits || !pos_logp || !pos_entropy || !seq_logp || !seq_entropy) return TPA_ERR_INVALID_ARG;
  if (vocab < 1 || row_stride < vocab || (row_stride & 7) || (reinterpret_cast<uintptr_t>(logits) & 15))
    return TPA_ERR_INVALID_ARG;
  if (layout != TPA_LOGITS_COMPACT && layout != TPA_LOGITS_PADDED) return TPA_ERR_INVALID_ARG;
  if (tree->n_trees < 1 || tree->t_pad < 1 || tree->n_seqs < 1) return TPA_ERR_INVALID_ARG;
  if (tree->max_token < 0 || tree->max_token >= vocab) return TPA_ERR_INVALID_ARG;  // a label past the row
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  row_kernel<<<dim3(tree->t_pad, tree->n_trees), kRowThreads, 0, st>>>(
      static_cast<const uint16_t*>(logits), row_stride, layout, vocab, tree->t_pad, tree->total_tree_tokens,
      tree->n_tokens, tree->tok_base, tree->tokens, tree->parent, tree->child_off, tree->child_pos, pos_logp,
      pos_entropy);
  TPA_CUDA_TRY(cudaGetLastError());
  return tpa_internal_seq_gather(tree, pos_logp, pos_entropy, seq_logp, seq_entropy, stream);
}

int tpa_internal_seq_gather(const tpa_tree_view* tree, const float* pos_logp, const float* pos_entropy,
                            float* seq_logp, float* seq_entropy, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  seq_gather_kernel<<<tree->n_seqs, 256, 0, st>>>(tree->t_pad, tree->n_trees, tree->total_seq_tokens,
                                                  tree->n_tokens, tree->seq_tree, tree->seq_off, tree->seq_pos,
                                                  pos_logp, pos_entropy, seq_logp, seq_entropy);
  TPA_CUDA_TRY(cudaGetLastError());
  return TPA_OK;
}
