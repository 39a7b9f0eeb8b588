// Tree attention backward on tcgen05 tensor cores (sm_103a).
//
// Gradients of <dO, O> for the tree attention forward (tree training page,
// §树构建过程 mask caption: query i sees key j iff j <= i <= E[j]):
//   P_ij = exp(scale q_i.k_j - LSE_i),   D_i = dO_i . O_i
//   dV_j = sum_i P_ij dO_i,   dS_ij = P_ij (dO_i . v_j - D_i)
//   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i
// with dK/dV summed over the query heads of each key/value head.
//
// Kernels: (1) preprocess: D = rowsum(dO * O) in fp32 and a zeroed fp32 dQ
// accumulator (the caller's dQ buffer itself for fp32 gradients); (2) main:
// one CTA per (key tile, kv head, tree) walks the non-empty query tiles of
// its key tile (per-key-block CSR) for every query head of the group;
// (3) bf16 gradients only: dQ accumulator -> bf16.
//
// Main-kernel roles (192 threads):
//   warp 4  TMA producer: K, V once; per step Q, dO (+ LSE, D rows);
//   warp 5  MMA issuer: S^T = K Q^T and dP^T = V dO^T into TMEM, then
//           dV += P^T dO, dK += dS^T Q, dQ = dS K (the dS^T tile in shared
//           memory read once K-major and once MN-major);
//   warps 0-3: thread r owns key row r for P^T / dS^T (TMEM lanes = keys),
//           then reads the dQ tile (TMEM lanes = queries) and adds it into
//           the fp32 accumulator with 16-byte vector reductions.
// TMEM: S^T / dQ cols [0,128), dP^T [128,256), dV [256,256+d), dK [256+d, 256+2d).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

int tpa_internal_check_attn_args(const tpa_tree_view* tree, const tpa_blockmask_view* mask, int hq,
                                 int hkv, int d);

namespace {

__device__ unsigned int g_status_bwd = 0;

constexpr int kB = 128;
constexpr uint32_t kChunk = 128 * 128;
constexpr float kLog2e = 1.4426950408889634f;

struct BwdParams {
  const float* lse;     // [B, Hq, T]
  const float* dvec;    // D, [B, Hq, T]
  float* dq_acc;        // [B, T, Hq, d] fp32 (the dQ output itself when gradients are fp32)
  void* dk;             // [B, T, Hkv, d], fp32 or bf16
  void* dv;
  const int32_t* subtree_end;
  const int32_t* n_tokens;
  const int32_t* k_ptr;
  const int32_t* k_idx;
  int32_t t_pad, n_blk, cap, hq, hkv;
  float scale, scale_log2;
};

template <int D>
struct BwdCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + NCH * kChunk;
  static constexpr uint32_t OFF_Q = OFF_V + NCH * kChunk;
  static constexpr uint32_t OFF_DO = OFF_Q + NCH * kChunk;
  static constexpr uint32_t OFF_PT = OFF_DO + NCH * kChunk;
  static constexpr uint32_t OFF_DST = OFF_PT + 2 * kChunk;
  static constexpr uint32_t OFF_LSE = OFF_DST + 2 * kChunk;
  static constexpr uint32_t OFF_DV = OFF_LSE + kB * 4;
  static constexpr uint32_t OFF_BAR = OFF_DV + kB * 4;
  // kv_full, q_full, q_empty, s_full, p_ready, dq_full, tmem_free, drain
  static constexpr int NBAR = 8;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16 + 1024;
};

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

template <int D, bool F32OUT>
__global__ void __launch_bounds__(192, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdParams p) {
  using C = BwdCfg<D>;
  constexpr int NCH = C::NCH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sPT = smem + C::OFF_PT;
  uint8_t* sDST = smem + C::OFF_DST;
  float* sLSE = reinterpret_cast<float*>(smem + C::OFF_LSE);
  float* sDv = reinterpret_cast<float*>(smem + C::OFF_DV);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bar + 0;
  uint64_t* q_full = bar + 1;
  uint64_t* q_empty = bar + 2;
  uint64_t* s_full = bar + 3;
  uint64_t* p_ready = bar + 4;
  uint64_t* dq_full = bar + 5;
  uint64_t* tmem_free = bar + 6;
  uint64_t* drain = bar + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, g = blockIdx.y, kb = blockIdx.x;
  const int G = p.hq / p.hkv;
  const int32_t* kp = p.k_ptr + b * (p.n_blk + 1);
  const int n_col = kp[kb + 1] - kp[kb];
  const int32_t* list = p.k_idx + int64_t(b) * p.cap + kp[kb];
  const int n_steps = G * n_col;
  const int krow = b * p.t_pad + kb * kB;

  if (threadIdx.x == 0) {
    tc::mbar_init(kv_full, 1);
    tc::mbar_init(q_full, 1);
    tc::mbar_init(q_empty, 1);
    tc::mbar_init(s_full, 1);
    tc::mbar_init(p_ready, 128);
    tc::mbar_init(dq_full, 1);
    tc::mbar_init(tmem_free, 128);
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
    if (lane == 0 && n_steps > 0) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      tc::tma_prefetch_desc(&tm_do);
      tc::mbar_arrive_expect_tx(kv_full, 2 * NCH * kChunk);
      for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sK + c * kChunk, &tm_k, kv_full, c * 64, g, krow);
      for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sV + c * kChunk, &tm_v, kv_full, c * 64, g, krow);
      int step = 0;
      for (; step < n_steps; ++step) {
        if (!tc::mbar_wait(q_empty, (step & 1) ^ 1, abort_flag, &g_status_bwd)) break;
        const int h = g * G + step / n_col;
        const int qb = list[step % n_col] >> 1;
        const int qrow = b * p.t_pad + qb * kB;
        const int64_t vec = (int64_t(b) * p.hq + h) * p.t_pad + qb * kB;
        tc::mbar_arrive_expect_tx(q_full, 2 * NCH * kChunk + 2 * kB * 4);
        for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sQ + c * kChunk, &tm_q, q_full, c * 64, h, qrow);
        for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sDO + c * kChunk, &tm_do, q_full, c * 64, h, qrow);
        tc::bulk_load(sLSE, p.lse + vec, kB * 4, q_full);
        tc::bulk_load(sDv, p.dvec + vec, kB * 4, q_full);
      }
      if (*abort_flag) {
        volatile int never = 0;
        tc::mbar_wait(kv_full, 0, &never, &g_status_bwd, 100000000ull);
        if (step > 0) tc::mbar_wait(q_full, (step - 1) & 1, &never, &g_status_bwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_kv = tc::idesc_bf16(128, D, false, true);
      constexpr uint32_t idesc_q = tc::idesc_bf16(128, D, true, true);
      const uint32_t aK = tc::smem_u32(sK), aV = tc::smem_u32(sV), aQ = tc::smem_u32(sQ),
                     aDO = tc::smem_u32(sDO), aPT = tc::smem_u32(sPT), aDST = tc::smem_u32(sDST);
      bool ok = tc::mbar_wait(kv_full, 0, abort_flag, &g_status_bwd);
      for (int step = 0; ok && step < n_steps; ++step) {
        if (!tc::mbar_wait(q_full, step & 1, abort_flag, &g_status_bwd)) break;
        if (!tc::mbar_wait(tmem_free, (step & 1) ^ 1, abort_flag, &g_status_bwd)) break;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {  // S^T = K Q^T
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          tc::mma_ss(tmem + 0, tc::smem_desc(aK + off, 16, 1024), tc::smem_desc(aQ + off, 16, 1024),
                     idesc_s, k > 0);
        }
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {  // dP^T = V dO^T
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          tc::mma_ss(tmem + 128, tc::smem_desc(aV + off, 16, 1024), tc::smem_desc(aDO + off, 16, 1024),
                     idesc_s, k > 0);
        }
        tc::mma_commit(s_full);
        if (!tc::mbar_wait(p_ready, step & 1, abort_flag, &g_status_bwd)) break;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < kB / 16; ++k) {  // dV += P^T dO ; dK += dS^T Q
          const uint32_t offa = (k >> 2) * kChunk + (k & 3) * 32;
          const uint32_t acc = (step > 0 || k > 0) ? 1u : 0u;
          tc::mma_ss(tmem + 256, tc::smem_desc(aPT + offa, 16, 1024),
                     tc::smem_desc(aDO + k * 2048, kChunk, 1024), idesc_kv, acc);
          tc::mma_ss(tmem + 256 + D, tc::smem_desc(aDST + offa, 16, 1024),
                     tc::smem_desc(aQ + k * 2048, kChunk, 1024), idesc_kv, acc);
        }
#pragma unroll
        for (int k = 0; k < kB / 16; ++k)  // dQ = dS K
          tc::mma_ss(tmem + 0, tc::smem_desc(aDST + k * 2048, kChunk, 1024),
                     tc::smem_desc(aK + k * 2048, kChunk, 1024), idesc_q, k > 0);
        tc::mma_commit(q_empty);
        tc::mma_commit(dq_full);
      }
      if (*abort_flag) {
        volatile int never = 0;
        tc::mma_commit(drain);
        tc::mbar_wait(drain, 0, &never, &g_status_bwd, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps
    const int r = threadIdx.x;
    const int j = kb * kB + r;  // key position owned by this thread
    const int n = p.n_tokens[b];
    const int Ej = (j < n) ? p.subtree_end[krow + r] : -1;
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    auto wait_all = [&](uint64_t* b_, uint32_t par) {
      return __all_sync(0xffffffffu, tc::mbar_wait(b_, par, abort_flag, &g_status_bwd));
    };
    bool ok = true;
    for (int step = 0; step < n_steps; ++step) {
      const int h = g * G + step / n_col;
      const int entry = list[step % n_col];
      const int qb = entry >> 1;
      const bool full = entry & 1;
      if (!wait_all(q_full, step & 1) || !wait_all(s_full, step & 1)) { ok = false; break; }
      tc::tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t sv[32], dpv[32];
        tc::tmem_ld32(tmem + lane_base + cc * 32, sv);
        tc::tmem_ld32(tmem + lane_base + 128 + cc * 32, dpv);
        tc::tmem_ld_wait();
        uint32_t pw[16], dw[16];
#pragma unroll
        for (int u = 0; u < 32; u += 2) {
          float pp[2], ds[2];
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            const int c = cc * 32 + u + w;
            const int qi = qb * kB + c;
            const bool vis = full || (j <= qi && qi <= Ej);
            const float pe = tc::ex2(fmaf(__uint_as_float(sv[u + w]), p.scale_log2, -sLSE[c] * kLog2e));
            pp[w] = vis ? pe : 0.f;
            ds[w] = pp[w] * (__uint_as_float(dpv[u + w]) - sDv[c]);
          }
          pw[u >> 1] = tc::pack_bf16(pp[0], pp[1]);
          dw[u >> 1] = tc::pack_bf16(ds[0], ds[1]);
        }
        uint8_t* rowP = sPT + (cc >> 1) * kChunk;
        uint8_t* rowS = sDST + (cc >> 1) * kChunk;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const uint32_t o = tc::sw128_offset(r, (cc & 1) * 4 + t);
          *reinterpret_cast<uint4*>(rowP + o) = make_uint4(pw[4 * t], pw[4 * t + 1], pw[4 * t + 2], pw[4 * t + 3]);
          *reinterpret_cast<uint4*>(rowS + o) = make_uint4(dw[4 * t], dw[4 * t + 1], dw[4 * t + 2], dw[4 * t + 3]);
        }
      }
      tc::fence_proxy_async_smem();
      tc::tc_fence_before();
      tc::mbar_arrive(p_ready);

      if (!wait_all(dq_full, step & 1)) { ok = false; break; }
      tc::tc_fence_after();
      const int qi = qb * kB + r;  // dQ tile: TMEM lane = query row
      float* dst = p.dq_acc + ((int64_t(b) * p.t_pad + qi) * p.hq + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t v[32];
        tc::tmem_ld32(tmem + lane_base + c * 32, v);
        tc::tmem_ld_wait();
        if (qi < n) {
#pragma unroll
          for (int t = 0; t < 8; ++t)
            red_add_v4(dst + c * 32 + 4 * t, __uint_as_float(v[4 * t]) * p.scale,
                       __uint_as_float(v[4 * t + 1]) * p.scale, __uint_as_float(v[4 * t + 2]) * p.scale,
                       __uint_as_float(v[4 * t + 3]) * p.scale);
        }
      }
      tc::tc_fence_before();
      tc::mbar_arrive(tmem_free);
    }
    // dK, dV rows of this key tile
    constexpr int ESZ = F32OUT ? 4 : 2;
    uint8_t* dk_row = static_cast<uint8_t*>(p.dk) + (int64_t(krow + r) * p.hkv + g) * D * ESZ;
    uint8_t* dv_row = static_cast<uint8_t*>(p.dv) + (int64_t(krow + r) * p.hkv + g) * D * ESZ;
    if (n_steps == 0) {
      const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < D * ESZ / 16; ++c) {
        reinterpret_cast<uint4*>(dk_row)[c] = z;
        reinterpret_cast<uint4*>(dv_row)[c] = z;
      }
    } else if (ok && F32OUT) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t vv[32], kk[32];
        tc::tmem_ld32(tmem + lane_base + 256 + c * 32, vv);
        tc::tmem_ld32(tmem + lane_base + 256 + D + c * 32, kk);
        tc::tmem_ld_wait();
        uint4* dV4 = reinterpret_cast<uint4*>(dv_row + c * 128);
        uint4* dK4 = reinterpret_cast<uint4*>(dk_row + c * 128);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          dV4[t] = make_uint4(vv[4 * t], vv[4 * t + 1], vv[4 * t + 2], vv[4 * t + 3]);
          dK4[t] = make_uint4(__float_as_uint(__uint_as_float(kk[4 * t]) * p.scale),
                              __float_as_uint(__uint_as_float(kk[4 * t + 1]) * p.scale),
                              __float_as_uint(__uint_as_float(kk[4 * t + 2]) * p.scale),
                              __float_as_uint(__uint_as_float(kk[4 * t + 3]) * p.scale));
        }
      }
    } else if (ok) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t vv[32], kk[32];
        tc::tmem_ld32(tmem + lane_base + 256 + c * 32, vv);
        tc::tmem_ld32(tmem + lane_base + 256 + D + c * 32, kk);
        tc::tmem_ld_wait();
        uint32_t wv[16], wk[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          wv[u] = tc::pack_bf16(__uint_as_float(vv[2 * u]), __uint_as_float(vv[2 * u + 1]));
          wk[u] = tc::pack_bf16(__uint_as_float(kk[2 * u]) * p.scale, __uint_as_float(kk[2 * u + 1]) * p.scale);
        }
        uint4* dV4 = reinterpret_cast<uint4*>(dv_row + c * 64);
        uint4* dK4 = reinterpret_cast<uint4*>(dk_row + c * 64);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          dV4[t] = make_uint4(wv[4 * t], wv[4 * t + 1], wv[4 * t + 2], wv[4 * t + 3]);
          dK4[t] = make_uint4(wk[4 * t], wk[4 * t + 1], wk[4 * t + 2], wk[4 * t + 3]);
        }
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 5) tc::tmem_dealloc(tmem, 512);
}

// D[b, h, i] = sum_d dO * O (fp32) for real rows, 0 for pad rows; one warp per
// (b, i, h) row.  Also zeroes the fp32 dQ accumulator.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      const int32_t* __restrict__ n_tokens, int32_t t_pad,
                                                      int32_t hq, int64_t n_rows, float* __restrict__ dvec,
                                                      float* __restrict__ dq_acc) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < n_rows; row += warps) {
    const int h = int(row % hq);
    const int64_t bt = row / hq;
    const int b = int(bt / t_pad), i = int(bt % t_pad);
    float s = 0.f;
    if (i < n_tokens[b]) {
      constexpr int PER = D / 32;  // elements per lane
      const __nv_bfloat16* a = o + row * D + lane * PER;
      const __nv_bfloat16* c = dout + row * D + lane * PER;
#pragma unroll
      for (int e = 0; e < PER; ++e) s += __bfloat162float(a[e]) * __bfloat162float(c[e]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    }
    if (lane == 0) dvec[(int64_t(b) * hq + h) * t_pad + i] = s;
  }
  float4* z = reinterpret_cast<float4*>(dq_acc);
  const int64_t n4 = n_rows * D / 4;
  for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < n4; k += int64_t(gridDim.x) * blockDim.x)
    z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
}

__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc,
                                                         __nv_bfloat16* __restrict__ dq, int64_t n8) {
  for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < n8; k += int64_t(gridDim.x) * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * k];
    const float4 c = reinterpret_cast<const float4*>(acc)[2 * k + 1];
    reinterpret_cast<uint4*>(dq)[k] = make_uint4(tc::pack_bf16(a.x, a.y), tc::pack_bf16(a.z, a.w),
                                                 tc::pack_bf16(c.x, c.y), tc::pack_bf16(c.z, c.w));
  }
}

inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

int grid_for(int64_t work, int per_block) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = (work + per_block - 1) / per_block;
  const int64_t cap = int64_t(sms) * 8;
  return int(want < 1 ? 1 : (want > cap ? cap : want));
}

template <int D, bool F32OUT>
int launch_bwd(const tpa_tree_view* tree, const tpa_blockmask_view* mask, const void* q, const void* k,
               const void* v, const void* o, const float* lse, const void* dout, void* dq, void* dk,
               void* dv, void* ws, int hq, int hkv, float scale, cudaStream_t st) {
  const int64_t rows = int64_t(tree->n_trees) * tree->t_pad;
  // workspace: D [B, Hq, T] fp32, then (bf16 gradients only) the fp32 dQ accumulator
  float* dvec = static_cast<float*>(ws);
  float* dq_acc = F32OUT ? static_cast<float*>(dq)
                         : reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + align256(uint64_t(rows) * hq * 4));
  const int64_t n_rows = rows * hq;
  bwd_pre_kernel<D><<<grid_for(n_rows * 32, 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), tree->n_tokens,
      tree->t_pad, hq, n_rows, dvec, dq_acc);
  TPA_CUDA_TRY(cudaGetLastError());

  CUtensorMap tq, tk, tv, tdo;
  if (!tmap::make_rows_heads_d(&tq, q, rows, hq, D) || !tmap::make_rows_heads_d(&tk, k, rows, hkv, D) ||
      !tmap::make_rows_heads_d(&tv, v, rows, hkv, D) || !tmap::make_rows_heads_d(&tdo, dout, rows, hq, D))
    return TPA_ERR_CUDA;
  BwdParams prm;
  prm.lse = lse;
  prm.dvec = dvec;
  prm.dq_acc = dq_acc;
  prm.dk = dk;
  prm.dv = dv;
  prm.subtree_end = tree->subtree_end;
  prm.n_tokens = tree->n_tokens;
  prm.k_ptr = mask->k_ptr;
  prm.k_idx = mask->k_idx;
  prm.t_pad = tree->t_pad;
  prm.n_blk = mask->n_blk;
  prm.cap = mask->cap;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.scale = scale;
  prm.scale_log2 = scale * kLog2e;
  const uint32_t smem = BwdCfg<D>::BYTES;
  TPA_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_kernel<D, F32OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
  attn_bwd_kernel<D, F32OUT><<<dim3(mask->n_blk, hkv, tree->n_trees), 192, smem, st>>>(tq, tk, tv, tdo, prm);
  TPA_CUDA_TRY(cudaGetLastError());
  if (F32OUT) return TPA_OK;

  const int64_t n8 = n_rows * D / 8;
  dq_convert_kernel<<<grid_for(n8, 256), 256, 0, st>>>(dq_acc, static_cast<__nv_bfloat16*>(dq), n8);
  TPA_CUDA_TRY(cudaGetLastError());
  return TPA_OK;
}

}  // namespace

TPA_DEFINE_STATUS_READER(tpa_internal_status_bwd, g_status_bwd)

extern "C" uint64_t tpa_tree_attn_bwd_workspace_bytes(int32_t n_trees, int32_t t_pad, int32_t n_heads_q,
                                                      int32_t head_dim, int32_t grad_dtype) {
  if (n_trees < 1 || t_pad < 1 || n_heads_q < 1 || head_dim < 1) return 0;
  if (grad_dtype != TPA_GRAD_F32 && grad_dtype != TPA_GRAD_BF16) return 0;
  const uint64_t rows = uint64_t(n_trees) * uint64_t(t_pad);
  const uint64_t dvec = align256(rows * n_heads_q * 4);
  return grad_dtype == TPA_GRAD_F32 ? dvec : dvec + align256(rows * n_heads_q * head_dim * 4);
}

extern "C" int tpa_tree_attn_bwd(const tpa_tree_view* tree, const tpa_blockmask_view* mask, const void* q,
                                 const void* k, const void* v, const void* o, const float* lse,
                                 const void* dout, void* dq, void* dk, void* dv, void* workspace,
                                 uint64_t workspace_bytes, int32_t n_heads_q, int32_t n_heads_kv,
                                 int32_t head_dim, float softmax_scale, int32_t grad_dtype, void* stream) {
  const int rc = tpa_internal_check_attn_args(tree, mask, n_heads_q, n_heads_kv, head_dim);
  if (rc != TPA_OK) return rc;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !workspace) return TPA_ERR_INVALID_ARG;
  const uintptr_t al = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o) |
                       reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
                       reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv) |
                       reinterpret_cast<uintptr_t>(lse);
  if ((al & 15) || (reinterpret_cast<uintptr_t>(workspace) & 255)) return TPA_ERR_INVALID_ARG;
  if (grad_dtype != TPA_GRAD_F32 && grad_dtype != TPA_GRAD_BF16) return TPA_ERR_INVALID_ARG;
  if (workspace_bytes <
      tpa_tree_attn_bwd_workspace_bytes(tree->n_trees, tree->t_pad, n_heads_q, head_dim, grad_dtype))
    return TPA_ERR_BUFFER_TOO_SMALL;
  const float scale = softmax_scale > 0.f ? softmax_scale : 1.0f / sqrtf(float(head_dim));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool f32 = grad_dtype == TPA_GRAD_F32;
#define TPA_BWD_ARGS tree, mask, q, k, v, o, lse, dout, dq, dk, dv, workspace, n_heads_q, n_heads_kv, scale, st
  if (head_dim == 128) return f32 ? launch_bwd<128, true>(TPA_BWD_ARGS) : launch_bwd<128, false>(TPA_BWD_ARGS);
  return f32 ? launch_bwd<64, true>(TPA_BWD_ARGS) : launch_bwd<64, false>(TPA_BWD_ARGS);
#undef TPA_BWD_ARGS
}

// ---------------------------------------------------------------------------
// Backward without a caller-provided workspace.
//
// Some callers cannot hand the library a device workspace: runtimes that
// reserve the whole device for their own pool and forbid further cudaMalloc
// calls, or plain-C integrations that have no allocator to draw from.  For
// them the backward's scratch (D = rowsum(dO * O), and the fp32 dQ
// accumulator when bf16 gradients are requested) lives in one fixed array
// compiled into this library.  Every GPU that loads the library keeps that
// array until the process exits.  Problems whose scratch does not fit are
// rejected with TPA_ERR_BUFFER_TOO_SMALL before any work is enqueued.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr uint64_t kNoAllocScratchBytes = 16ull << 20;  // 16 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The host-side
// name of a __device__ array is only a stand-in, so the address is looked up
// once per device (with that device current) and cached.
int noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return TPA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return TPA_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();
      return TPA_ERR_CUDA;
    }
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return TPA_OK;
}

}  // namespace

extern "C" int tpa_tree_attn_bwd_noalloc(const tpa_tree_view* tree, const tpa_blockmask_view* mask,
                                         const void* q, const void* k, const void* v, const void* o,
                                         const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                         int32_t n_heads_q, int32_t n_heads_kv, int32_t head_dim,
                                         float softmax_scale, int32_t grad_dtype, void* stream) {
  if (!tree) return TPA_ERR_INVALID_ARG;
  const uint64_t need =
      tpa_tree_attn_bwd_workspace_bytes(tree->n_trees, tree->t_pad, n_heads_q, head_dim, grad_dtype);
  if (need == 0) return TPA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return TPA_ERR_BUFFER_TOO_SMALL;
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != TPA_OK) return rc;
  return tpa_tree_attn_bwd(tree, mask, q, k, v, o, lse, dout, dq, dk, dv, scratch, kNoAllocScratchBytes,
                           n_heads_q, n_heads_kv, head_dim, softmax_scale, grad_dtype, stream);
}
