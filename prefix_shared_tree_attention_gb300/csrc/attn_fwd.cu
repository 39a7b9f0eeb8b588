// Tree attention forward on tcgen05 tensor cores (sm_103a).
//
// Semantics (tree training page, §树构建过程 mask caption, §注意力机制): query
// i of a packed tree sees key j iff j <= i <= E[j] (j is i or an ancestor);
// O_i = softmax over the visible keys of scale * q_i.k_j, times v_j.
// Only non-empty 128x128 tiles are visited (the per-query-block CSR from the
// classifier); the ancestor test runs only on PARTIAL tiles.
//
// One CTA = one 128-query tile of one query head.  Warp roles:
//   warp 4  TMA producer: Q once, then K/V tiles (+ E of the key tile) into an
//           NS-stage ring;
//   warp 5  MMA issuer (one thread): S = Q K^T into a double-buffered TMEM
//           tile, then O += P V with O resident in TMEM;
//   warps 0-3 softmax: thread r owns query row r (= TMEM lane r); fp32 online
//           softmax in the log2 domain, P written to shared memory as bf16 in
//           the 128-byte-swizzled K-major layout the MMA reads; O is rescaled
//           in TMEM only when the running max grows by more than 2^8 (exact:
//           numerator and denominator share the stale max).
// TMEM: S0 cols [0,128), S1 [128,256), O [256, 256+d).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace {

__device__ unsigned int g_status_fwd = 0;

constexpr int kB = 128;
constexpr uint32_t kChunk = 128 * 128;  // bytes of a 128-row x 64-col bf16 tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  const int32_t* subtree_end;
  const int32_t* n_tokens;
  const int32_t* q_ptr;
  const int32_t* q_idx;
  int32_t t_pad, n_blk, cap, hq, hkv;
  float scale_log2;  // softmax scale * log2(e)
};

template <int D>
struct FwdCfg {
  static constexpr int NCH = D / 64;
  static constexpr int NS = (D == 128) ? 2 : 3;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NCH * kChunk;
  static constexpr uint32_t OFF_V = OFF_K + NS * NCH * kChunk;
  static constexpr uint32_t OFF_P = OFF_V + NS * NCH * kChunk;
  static constexpr uint32_t OFF_E = OFF_P + 2 * kChunk;
  static constexpr uint32_t OFF_BAR = OFF_E + NS * kB * 4;
  // barriers: q_full, kv_full[NS], kv_empty[NS], s_full[2], s_free[2], p_full, o_done, drain
  static constexpr int NBAR = 1 + 2 * NS + 2 + 2 + 3;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
};

template <int D>
__global__ void __launch_bounds__(192, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D>;
  constexpr int NCH = C::NCH, NS = C::NS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sP = smem + C::OFF_P;
  int32_t* sE = reinterpret_cast<int32_t*>(smem + C::OFF_E);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bar;
  uint64_t* kv_full = bar + 1;
  uint64_t* kv_empty = bar + 1 + NS;
  uint64_t* s_full = bar + 1 + 2 * NS;
  uint64_t* s_free = bar + 3 + 2 * NS;
  uint64_t* p_full = bar + 5 + 2 * NS;
  uint64_t* o_done = bar + 6 + 2 * NS;
  uint64_t* drain = bar + 7 + 2 * NS;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y;
  const int qb = p.n_blk - 1 - blockIdx.x;  // deepest (usually heaviest) query blocks first
  const int g = h / (p.hq / p.hkv);
  const int n_it = p.q_ptr[b * (p.n_blk + 1) + qb + 1] - p.q_ptr[b * (p.n_blk + 1) + qb];
  const int32_t* list = p.q_idx + int64_t(b) * p.cap + p.q_ptr[b * (p.n_blk + 1) + qb];
  const int row0 = b * p.t_pad + qb * kB;  // global row of the tile's first query

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(kv_full + s, 1);
      tc::mbar_init(kv_empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(s_full + s, 1);
      tc::mbar_init(s_free + s, 128);
    }
    tc::mbar_init(p_full, 128);
    tc::mbar_init(o_done, 1);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 5) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_it > 0) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      tc::mbar_arrive_expect_tx(q_full, NCH * kChunk);
      for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sQ + c * kChunk, &tm_q, q_full, c * 64, h, row0);
      int it = 0;
      for (; it < n_it; ++it) {
        const int s = it % NS;
        if (!tc::mbar_wait(kv_empty + s, ((it / NS) & 1) ^ 1, abort_flag, &g_status_fwd)) break;
        const int kb = list[it] >> 1;
        const int krow = b * p.t_pad + kb * kB;
        tc::mbar_arrive_expect_tx(kv_full + s, 2 * NCH * kChunk + kB * 4);
        for (int c = 0; c < NCH; ++c)
          tc::tma_load_3d(sK + (s * NCH + c) * kChunk, &tm_k, kv_full + s, c * 64, g, krow);
        for (int c = 0; c < NCH; ++c)
          tc::tma_load_3d(sV + (s * NCH + c) * kChunk, &tm_v, kv_full + s, c * 64, g, krow);
        tc::bulk_load(sE + s * kB, p.subtree_end + krow, kB * 4, kv_full + s);
      }
      // On an abort, let the copies already issued land before the CTA exits.
      if (*abort_flag) {
        volatile int never = 0;
        for (int j = (it > NS ? it - NS : 0); j < it; ++j)
          tc::mbar_wait(kv_full + (j % NS), (j / NS) & 1, &never, &g_status_fwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_it > 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(128, D, false, true);
      const uint32_t aQ = tc::smem_u32(sQ), aK = tc::smem_u32(sK), aV = tc::smem_u32(sV),
                     aP = tc::smem_u32(sP);
      bool ok = tc::mbar_wait(q_full, 0, abort_flag, &g_status_fwd);
      for (int it = 0; ok && it <= n_it; ++it) {
        if (it < n_it) {
          const int s = it % NS, sb = it & 1;
          if (!tc::mbar_wait(kv_full + s, (it / NS) & 1, abort_flag, &g_status_fwd)) break;
          if (!tc::mbar_wait(s_free + sb, ((it >> 1) & 1) ^ 1, abort_flag, &g_status_fwd)) break;
          tc::tc_fence_after();
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
            const uint64_t da = tc::smem_desc(aQ + off, 16, 1024);
            const uint64_t db = tc::smem_desc(aK + s * NCH * kChunk + off, 16, 1024);
            tc::mma_ss(tmem + sb * 128, da, db, idesc_qk, k > 0);
          }
          tc::mma_commit(s_full + sb);
        }
        if (it >= 1) {
          const int j = it - 1, sj = j % NS;
          if (!tc::mbar_wait(p_full, j & 1, abort_flag, &g_status_fwd)) break;
          tc::tc_fence_after();
#pragma unroll
          for (int k = 0; k < kB / 16; ++k) {
            const uint64_t da = tc::smem_desc(aP + (k >> 2) * kChunk + (k & 3) * 32, 16, 1024);
            const uint64_t db = tc::smem_desc(aV + sj * NCH * kChunk + k * 2048, kChunk, 1024);
            tc::mma_ss(tmem + 256, da, db, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
          }
          tc::mma_commit(kv_empty + sj);
          tc::mma_commit(o_done);
        }
      }
      if (*abort_flag) {  // let issued MMAs finish before TMEM is released
        volatile int never = 0;
        tc::mma_commit(drain);
        tc::mbar_wait(drain, 0, &never, &g_status_fwd, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // query row within the tile = TMEM lane
    const int i = qb * kB + r;  // query position in the tree
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    __nv_bfloat16* orow = p.o + (int64_t(row0 + r) * p.hq + h) * D;
    float* lse_out = p.lse + (int64_t(b) * p.hq + h) * p.t_pad + i;
    // every lane waits, and the warp proceeds only if all lanes succeeded
    auto wait_all = [&](uint64_t* b_, uint32_t par) {
      return __all_sync(0xffffffffu, tc::mbar_wait(b_, par, abort_flag, &g_status_fwd));
    };
    if (n_it == 0) {
      const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
      *lse_out = 0.f;
    } else {
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      for (int it = 0; it < n_it; ++it) {
        const int sb = it & 1, s = it % NS;
        const int entry = list[it];
        const int kb = entry >> 1;
        const bool full = entry & 1;
        if (!wait_all(s_full + sb, (it >> 1) & 1)) { ok = false; break; }
        if (!wait_all(kv_full + s, (it / NS) & 1)) { ok = false; break; }
        tc::tc_fence_after();
        uint32_t sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tc::tmem_ld32(tmem + lane_base + sb * 128 + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sv + c * 32));
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(s_free + sb);

        float x[128];
        float mx = -INFINITY;
        if (full) {
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            x[c] = __uint_as_float(sv[c]) * p.scale_log2;
            mx = fmaxf(mx, x[c]);
          }
        } else {
          const int32_t* e = sE + s * kB;
          const int j0 = kb * kB;
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const bool vis = (j0 + c <= i) && (i <= e[c]);
            x[c] = vis ? __uint_as_float(sv[c]) * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, x[c]);
          }
        }
        const float m_new = fmaxf(m_run, mx);
        const bool resc = m_new > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
          alpha = tc::ex2(m_run - m_new);
          m_run = m_new;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        float sum = 0.f;
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float p0 = tc::ex2(x[2 * c] - m_use);
          const float p1 = tc::ex2(x[2 * c + 1] - m_use);
          sum += p0 + p1;
          pk[c] = tc::pack_bf16(p0, p1);
        }
        l_run = l_run * alpha + sum;

        if (it >= 1) {
          if (!wait_all(o_done, (it - 1) & 1)) { ok = false; break; }
          tc::tc_fence_after();
          if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t ov[32];
              tc::tmem_ld32(tmem + lane_base + 256 + c * 32, ov);
              tc::tmem_ld_wait();
#pragma unroll
              for (int u = 0; u < 32; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * alpha);
              tc::tmem_st32(tmem + lane_base + 256 + c * 32, ov);
            }
            tc::tmem_st_wait();
          }
        }
        // P row r -> two 128x64 swizzled chunks (keys 0-63, 64-127)
#pragma unroll
        for (int kc = 0; kc < 16; ++kc) {
          uint4 v = make_uint4(pk[4 * kc], pk[4 * kc + 1], pk[4 * kc + 2], pk[4 * kc + 3]);
          *reinterpret_cast<uint4*>(sP + (kc >> 3) * kChunk + tc::sw128_offset(r, kc & 7)) = v;
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        tc::mbar_arrive(p_full);
      }
      if (ok && wait_all(o_done, (n_it - 1) & 1)) {
        tc::tc_fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tc::tmem_ld32(tmem + lane_base + 256 + c * 32, ov);
          tc::tmem_ld_wait();
          uint32_t w[16];
#pragma unroll
          for (int u = 0; u < 16; ++u)
            w[u] = tc::pack_bf16(__uint_as_float(ov[2 * u]) * inv, __uint_as_float(ov[2 * u + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          dst[2] = make_uint4(w[8], w[9], w[10], w[11]);
          dst[3] = make_uint4(w[12], w[13], w[14], w[15]);
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        *lse_out = l_run > 0.f ? (m_use + __log2f(l_run)) * kLn2 : 0.f;
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 5) tc::tmem_dealloc(tmem, 512);
}

template <int D>
int launch_fwd(const tpa_tree_view* tree, const tpa_blockmask_view* mask, const void* q,
               const void* k, const void* v, void* o, float* lse, int hq, int hkv, float scale,
               cudaStream_t st) {
  const uint64_t rows = uint64_t(tree->n_trees) * tree->t_pad;
  CUtensorMap tq, tk, tv;
  if (!tmap::make_rows_heads_d(&tq, q, rows, hq, D) || !tmap::make_rows_heads_d(&tk, k, rows, hkv, D) ||
      !tmap::make_rows_heads_d(&tv, v, rows, hkv, D))
    return TPA_ERR_CUDA;
  FwdParams prm;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.subtree_end = tree->subtree_end;
  prm.n_tokens = tree->n_tokens;
  prm.q_ptr = mask->q_ptr;
  prm.q_idx = mask->q_idx;
  prm.t_pad = tree->t_pad;
  prm.n_blk = mask->n_blk;
  prm.cap = mask->cap;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.scale_log2 = scale * kLog2e;
  const uint32_t smem = FwdCfg<D>::BYTES;
  TPA_CUDA_TRY(cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  attn_fwd_kernel<D><<<dim3(mask->n_blk, hq, tree->n_trees), 192, smem, st>>>(tq, tk, tv, prm);
  TPA_CUDA_TRY(cudaGetLastError());
  return TPA_OK;
}

}  // namespace

TPA_DEFINE_STATUS_READER(tpa_internal_status_fwd, g_status_fwd)

int tpa_internal_check_attn_args(const tpa_tree_view* tree, const tpa_blockmask_view* mask, int hq,
                                 int hkv, int d) {
  if (!tree || !mask || !tree->subtree_end || !tree->n_tokens || !mask->q_ptr || !mask->q_idx ||
      !mask->k_ptr || !mask->k_idx)
    return TPA_ERR_INVALID_ARG;
  if (tree->n_trees < 1 || tree->n_trees > 65535 || tree->t_pad < kB || tree->t_pad % kB || mask->n_trees != tree->n_trees ||
      mask->n_blk != tree->t_pad / kB)
    return TPA_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || hq < 1 || hkv < 1 || hq % hkv != 0 || hq > 65535) return TPA_ERR_INVALID_ARG;
  if (uint64_t(tree->n_trees) * tree->t_pad > (uint64_t(1) << 31)) return TPA_ERR_INVALID_ARG;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return TPA_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return TPA_ERR_UNSUPPORTED_DEVICE;
  return TPA_OK;
}

extern "C" int tpa_tree_attn_fwd(const tpa_tree_view* tree, const tpa_blockmask_view* mask,
                                 const void* q, const void* k, const void* v, void* o, float* lse,
                                 int32_t n_heads_q, int32_t n_heads_kv, int32_t head_dim,
                                 float softmax_scale, void* stream) {
  const int rc = tpa_internal_check_attn_args(tree, mask, n_heads_q, n_heads_kv, head_dim);
  if (rc != TPA_OK) return rc;
  if (!q || !k || !v || !o || !lse) return TPA_ERR_INVALID_ARG;
  const uintptr_t al = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
  if ((al & 15) || (reinterpret_cast<uintptr_t>(lse) & 3)) return TPA_ERR_INVALID_ARG;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(float(head_dim));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return head_dim == 128 ? launch_fwd<128>(tree, mask, q, k, v, o, lse, n_heads_q, n_heads_kv, scale, st)
                         : launch_fwd<64>(tree, mask, q, k, v, o, lse, n_heads_q, n_heads_kv, scale, st);
}
