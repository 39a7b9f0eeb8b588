// Tree attention backward on tcgen05 tensor cores (sm_103a).
//
// Gradients of <dO, O> for the tree attention forward (tree training page,
// §树构建过程 mask caption: query i sees key j iff j <= i <= E[j]):
//   P_ij = exp(scale q_i.k_j - LSE_i),   D_i = dO_i . O_i
//   dV_j = sum_i P_ij dO_i,   dS_ij = P_ij (dO_i . v_j - D_i)
//   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i
// with dK/dV summed over the query heads of each key/value head.
//
// Three kernels, no atomics:
//  (1) preprocess: D = rowsum(dO * O) in fp32.
//  (2) KV kernel, one CTA per (key tile, kv head, tree): walks the non-empty
//      query tiles of its key tile (per-key-block CSR) for every query head of
//      the group and accumulates dK, dV in TMEM.  Per step the MMA issuer
//      runs S^T = K Q^T and dP^T = V dO^T; the four compute warpgroups (thread
//      r = key row r = TMEM lane r; warpgroup w = query columns [32w, 32w+32))
//      write P^T and dS^T back into TMEM as packed bf16 over the columns they
//      read, and the issuer runs dV += P^T dO and dK += dS^T Q with A read
//      from TMEM.  The next step's S^T / dP^T are issued right behind dK, so
//      the tensor core stays fed while the warpgroups compute.  A key only
//      sees the query interval [j, E[j]], applied on PARTIAL tiles.
//  (3) dQ kernel, one CTA per (query tile, query head, tree): walks the
//      query block's key tiles like the forward, recomputes S = Q K^T (double
//      buffered in TMEM) and dP = dO V^T, forms dS = P (dP - D) with the
//      forward's LSE and the precomputed partial-tile bit masks, writes dS as
//      packed bf16 into TMEM and accumulates dQ += dS K in TMEM; dQ is stored
//      once at the end.
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
constexpr uint32_t kChunk = 128 * 128;  // bytes of a 128-row x 64-col bf16 tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kSmemMax = 232448;   // 227 KB opt-in per CTA

struct BwdParams {
  const float* lse;     // [B, Hq, T]
  const float* dvec;    // D, [B, Hq, T]
  void* dq;             // [B, T, Hq, d], fp32 or bf16
  void* dk;             // [B, T, Hkv, d], fp32 or bf16
  void* dv;
  const int32_t* subtree_end;
  const int32_t* n_tokens;
  const int32_t* k_ptr;
  const int32_t* k_idx;
  const int32_t* q_ptr;
  const int32_t* q_idx;
  const uint4* qmask;
  int32_t t_pad, n_blk, cap, hq, hkv;
  float scale, scale_log2;
};

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Writes 16 fp32 values of one row as fp32 or bf16 (with a scale).
template <bool F32OUT>
__device__ __forceinline__ void store_row16(uint8_t* dst, const uint32_t (&v)[16], float scale) {
  if (F32OUT) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int t = 0; t < 4; ++t)
      d4[t] = make_uint4(__float_as_uint(__uint_as_float(v[4 * t]) * scale),
                         __float_as_uint(__uint_as_float(v[4 * t + 1]) * scale),
                         __float_as_uint(__uint_as_float(v[4 * t + 2]) * scale),
                         __float_as_uint(__uint_as_float(v[4 * t + 3]) * scale));
  } else {
    uint32_t w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      w[u] = tc::pack_bf16(__uint_as_float(v[2 * u]) * scale, __uint_as_float(v[2 * u + 1]) * scale);
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// =========================================================================== KV kernel

constexpr int kNWG = 4;                    // compute warpgroups per CTA
constexpr int kCW = kB / kNWG;             // columns per warpgroup (32)
constexpr int kThreads = 128 * kNWG + 64;  // + TMA warp + MMA warp
constexpr int kWTma = 4 * kNWG, kWMma = 4 * kNWG + 1;

// Packed bf16 A operand written by the warpgroups: warpgroup w owns columns
// [32w, 32w+32) of the region it read; P (or dS) for its 32 rows of K goes to
// the first 16 columns of that range (second-operand values to the last 16).
__device__ __forceinline__ uint32_t wg_a(uint32_t base, int k, uint32_t sub) {
  return base + 32 * (k >> 1) + sub + 8 * (k & 1);
}

template <int D>
struct KvCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = NCH * kChunk;
  static constexpr int NS_FIT = int((kSmemMax - 1024 - 2 * TILE - 4096) / (2 * TILE + 1024));
  static constexpr int NS = NS_FIT > 3 ? 3 : NS_FIT;  // Q/dO ring depth
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + TILE;
  static constexpr uint32_t OFF_Q = OFF_V + TILE;
  static constexpr uint32_t OFF_DO = OFF_Q + NS * TILE;
  static constexpr uint32_t OFF_LSE = OFF_DO + NS * TILE;   // NS x 128 fp32
  static constexpr uint32_t OFF_DV = OFF_LSE + NS * kB * 4; // NS x 128 fp32
  static constexpr uint32_t OFF_BAR = OFF_DV + NS * kB * 4;
  // kv_full, q_full[NS], q_empty[NS], s_full, dp_full, p_ready, ds_ready, drain
  static constexpr int NBAR = 1 + 2 * NS + 5;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16 + 1024;
  static_assert(NS >= 2, "shared memory budget");
  static_assert(BYTES <= kSmemMax, "shared memory budget");
};

template <int D, bool F32OUT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using C = KvCfg<D>;
  constexpr int NCH = C::NCH, NS = C::NS;
  constexpr uint32_t TILE = C::TILE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  float* sLSE = reinterpret_cast<float*>(smem + C::OFF_LSE);
  float* sDv = reinterpret_cast<float*>(smem + C::OFF_DV);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bar;
  uint64_t* q_full = bar + 1;
  uint64_t* q_empty = bar + 1 + NS;
  uint64_t* s_full = bar + 1 + 2 * NS;
  uint64_t* dp_full = s_full + 1;
  uint64_t* p_ready = s_full + 2;
  uint64_t* ds_ready = s_full + 3;
  uint64_t* drain = s_full + 4;
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
  constexpr uint32_t T_S = 0, T_DP = 128, T_DV = 256, T_DK = 256 + D;

  if (threadIdx.x == 0) {
    tc::mbar_init(kv_full, 1);
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(q_full + s, 1);
      tc::mbar_init(q_empty + s, 1);
    }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(dp_full, 1);
    tc::mbar_init(p_ready, 128 * kNWG);
    tc::mbar_init(ds_ready, 128 * kNWG);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kWMma) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWTma) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_steps > 0) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      tc::tma_prefetch_desc(&tm_do);
      tc::mbar_arrive_expect_tx(kv_full, 2 * TILE);
      for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sK + c * kChunk, &tm_k, kv_full, c * 64, g, krow);
      for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sV + c * kChunk, &tm_v, kv_full, c * 64, g, krow);
      int s = 0;
      for (; s < n_steps; ++s) {
        const int st = s % NS;
        if (!tc::mbar_wait(q_empty + st, ((s / NS) & 1) ^ 1, abort_flag, &g_status_bwd)) break;
        const int h = g * G + s / n_col;
        const int qb = list[s % n_col] >> 1;
        const int qrow = b * p.t_pad + qb * kB;
        const int64_t vec = (int64_t(b) * p.hq + h) * p.t_pad + qb * kB;
        tc::mbar_arrive_expect_tx(q_full + st, 2 * TILE + 2 * kB * 4);
        for (int c = 0; c < NCH; ++c)
          tc::tma_load_3d(sQ + st * TILE + c * kChunk, &tm_q, q_full + st, c * 64, h, qrow);
        for (int c = 0; c < NCH; ++c)
          tc::tma_load_3d(sDO + st * TILE + c * kChunk, &tm_do, q_full + st, c * 64, h, qrow);
        tc::bulk_load(sLSE + st * kB, p.lse + vec, kB * 4, q_full + st);
        tc::bulk_load(sDv + st * kB, p.dvec + vec, kB * 4, q_full + st);
      }
      if (*abort_flag) {  // let the copies already issued land before the CTA exits
        volatile int never = 0;
        tc::mbar_wait(kv_full, 0, &never, &g_status_bwd, 100000000ull);
        for (int j = (s > NS ? s - NS : 0); j < s; ++j)
          tc::mbar_wait(q_full + (j % NS), (j / NS) & 1, &never, &g_status_bwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kWMma) {
    // ------------------------------------------------------------ MMA issuer
    // Per step s: dV(s) as soon as P^T(s) is in TMEM, then S^T(s+1) into the
    // region P^T(s) came from (in order behind dV), then dK(s) once dS^T(s) is
    // in TMEM, then dP^T(s+1) into the region dS^T(s) came from.
    if (lane == 0 && n_steps > 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_kv = tc::idesc_bf16(128, D, false, true);
      const uint32_t aK = tc::smem_u32(sK), aV = tc::smem_u32(sV), aQ = tc::smem_u32(sQ),
                     aDO = tc::smem_u32(sDO);
      auto issue_s = [&](int s) {  // S^T = K Q^T
        const uint32_t qs = aQ + (s % NS) * TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          tc::mma_ss(tmem + T_S, tc::smem_desc(aK + off, 16, 1024), tc::smem_desc(qs + off, 16, 1024), idesc_s,
                     k > 0);
        }
        tc::mma_commit(s_full);
      };
      auto issue_dp = [&](int s) {  // dP^T = V dO^T
        const uint32_t dos = aDO + (s % NS) * TILE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          tc::mma_ss(tmem + T_DP, tc::smem_desc(aV + off, 16, 1024), tc::smem_desc(dos + off, 16, 1024),
                     idesc_s, k > 0);
        }
        tc::mma_commit(dp_full);
      };
      bool ok = tc::mbar_wait(kv_full, 0, abort_flag, &g_status_bwd) &&
                tc::mbar_wait(q_full, 0, abort_flag, &g_status_bwd);
      if (ok) {
        tc::tc_fence_after();
        issue_s(0);
        issue_dp(0);
      }
      for (int s = 0; ok && s < n_steps; ++s) {
        const int st = s % NS;
        const bool more = s + 1 < n_steps;
        const uint32_t qs = aQ + st * TILE, dos = aDO + st * TILE;
        if (!(ok = tc::mbar_wait(p_ready, s & 1, abort_flag, &g_status_bwd))) break;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < kB / 16; ++k)  // dV += P^T dO, P^T packed bf16 in TMEM
          mma_ts(tmem + T_DV, wg_a(tmem + T_S, k, 0), tc::smem_desc(dos + k * 2048, kChunk, 1024), idesc_kv,
                 (s > 0 || k > 0) ? 1u : 0u);
        if (more) {
          if (!(ok = tc::mbar_wait(q_full + (s + 1) % NS, ((s + 1) / NS) & 1, abort_flag, &g_status_bwd))) break;
          tc::tc_fence_after();
          issue_s(s + 1);
        }
        if (!(ok = tc::mbar_wait(ds_ready, s & 1, abort_flag, &g_status_bwd))) break;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < kB / 16; ++k)  // dK += dS^T Q, dS^T packed bf16 in TMEM
          mma_ts(tmem + T_DK, wg_a(tmem + T_DP, k, 0), tc::smem_desc(qs + k * 2048, kChunk, 1024), idesc_kv,
                 (s > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(q_empty + st);
        if (more)
          issue_dp(s + 1);
        else
          tc::mma_commit(s_full);  // final: dV and dK complete
      }
      if (*abort_flag) {  // let issued MMAs finish before TMEM is released
        volatile int never = 0;
        tc::mma_commit(drain);
        tc::mbar_wait(drain, 0, &never, &g_status_bwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp < 4 * kNWG) {
    // ------------------------------------------------------------ compute warpgroups
    const int w = warp >> 2;              // query columns [32w, 32w+32) of this warpgroup
    const int r = threadIdx.x & 127;      // key row = TMEM lane
    const int j = kb * kB + r;            // key position owned by this thread
    const int n = p.n_tokens[b];
    const int Ej = (j < n) ? p.subtree_end[krow + r] : -1;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    auto wait_all = [&](uint64_t* b_, uint32_t par) {
      return __all_sync(0xffffffffu, tc::mbar_wait(b_, par, abort_flag, &g_status_bwd));
    };
    bool ok = true;
    for (int s = 0; s < n_steps; ++s) {
      const int st = s % NS;
      const int entry = list[s % n_col];
      const int qb = entry >> 1;
      const bool full = entry & 1;
      if (!wait_all(q_full + st, (s / NS) & 1) || !wait_all(s_full, s & 1)) { ok = false; break; }
      tc::tc_fence_after();
      // ---- P^T = exp2(S * scale*log2e - LSE*log2e) on this group's 32 query columns
      float pf[kCW];
      {
        uint32_t sv[kCW];
        tc::tmem_ld32(tmem + lane_base + T_S + kCW * w, sv);
        const float4* l4 = reinterpret_cast<const float4*>(sLSE + st * kB + kCW * w);
        tc::tmem_ld_wait();
        const int lo = j - (qb * kB + kCW * w);  // visible query columns: [lo, hi]
        const int hi = Ej - (qb * kB + kCW * w);
#pragma unroll
        for (int c4 = 0; c4 < kCW / 4; ++c4) {
          const float4 l = l4[c4];
          const float lv[4] = {l.x, l.y, l.z, l.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int c = 4 * c4 + u;
            pf[c] = tc::ex2(fmaf(__uint_as_float(sv[c]), p.scale_log2, -lv[u] * kLog2e));
          }
        }
        if (!full) {
#pragma unroll
          for (int c = 0; c < kCW; ++c)
            if (c < lo || c > hi) pf[c] = 0.f;
        }
        uint32_t pw[kCW / 2];
#pragma unroll
        for (int u = 0; u < kCW / 2; ++u) pw[u] = tc::pack_bf16(pf[2 * u], pf[2 * u + 1]);
        tc::tmem_st16(tmem + lane_base + T_S + kCW * w, pw);  // over the first half of what was read
        tc::tmem_st_wait();
      }
      tc::tc_fence_before();
      tc::mbar_arrive(p_ready);
      // ---- dS^T = P^T (dP^T - D)
      if (!wait_all(dp_full, s & 1)) { ok = false; break; }
      tc::tc_fence_after();
      {
        uint32_t dpv[kCW];
        tc::tmem_ld32(tmem + lane_base + T_DP + kCW * w, dpv);
        const float4* d4 = reinterpret_cast<const float4*>(sDv + st * kB + kCW * w);
        tc::tmem_ld_wait();
        uint32_t dw[kCW / 2];
#pragma unroll
        for (int c4 = 0; c4 < kCW / 4; ++c4) {
          const float4 dd = d4[c4];
          const int c = 4 * c4;
          dw[2 * c4] = tc::pack_bf16(pf[c] * (__uint_as_float(dpv[c]) - dd.x),
                                     pf[c + 1] * (__uint_as_float(dpv[c + 1]) - dd.y));
          dw[2 * c4 + 1] = tc::pack_bf16(pf[c + 2] * (__uint_as_float(dpv[c + 2]) - dd.z),
                                         pf[c + 3] * (__uint_as_float(dpv[c + 3]) - dd.w));
        }
        tc::tmem_st16(tmem + lane_base + T_DP + kCW * w, dw);
        tc::tmem_st_wait();
      }
      tc::tc_fence_before();
      tc::mbar_arrive(ds_ready);
    }
    // ---- dK, dV rows of this key tile (warpgroup w: head-dim columns [w d/4, (w+1) d/4))
    constexpr int ESZ = F32OUT ? 4 : 2;
    constexpr int DW = D / kNWG;
    const int64_t off = ((int64_t(krow + r) * p.hkv + g) * D + w * DW) * ESZ;
    uint8_t* dk_row = static_cast<uint8_t*>(p.dk) + off;
    uint8_t* dv_row = static_cast<uint8_t*>(p.dv) + off;
    if (n_steps == 0) {
      const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < DW * ESZ / 16; ++c) {
        reinterpret_cast<uint4*>(dk_row)[c] = z;
        reinterpret_cast<uint4*>(dv_row)[c] = z;
      }
    } else if (ok && wait_all(s_full, n_steps & 1)) {
      tc::tc_fence_after();
#pragma unroll
      for (int c = 0; c < DW / 16; ++c) {
        uint32_t vv[16], kk[16];
        tc::tmem_ld16(tmem + lane_base + T_DV + w * DW + c * 16, vv);
        tc::tmem_ld16(tmem + lane_base + T_DK + w * DW + c * 16, kk);
        tc::tmem_ld_wait();
        store_row16<F32OUT>(dv_row + c * 16 * ESZ, vv, 1.f);
        store_row16<F32OUT>(dk_row + c * 16 * ESZ, kk, p.scale);
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kWMma) tc::tmem_dealloc(tmem, 512);
}

// =========================================================================== dQ kernel

template <int D>
struct DqCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = NCH * kChunk;
  static constexpr int NSK = 3;  // K ring (K(j) is read by S(j) and again by dQ(j))
  static constexpr int NSV = D == 128 ? 1 : 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = TILE;
  static constexpr uint32_t OFF_K = 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + NSK * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + NSV * TILE;
  // q_full, k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full[2], dp_full, dp_free,
  // ds_ready, dq_final, drain
  static constexpr int NBAR = 1 + 2 * NSK + 2 * NSV + 7;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16 + 1024;
  static_assert(BYTES <= kSmemMax, "shared memory budget");
};

template <int D, bool F32OUT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using C = DqCfg<D>;
  constexpr int NCH = C::NCH, NSK = C::NSK, NSV = C::NSV;
  constexpr uint32_t TILE = C::TILE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bar;
  uint64_t* k_full = bar + 1;
  uint64_t* k_empty = k_full + NSK;
  uint64_t* v_full = k_empty + NSK;
  uint64_t* v_empty = v_full + NSV;
  uint64_t* s_full = v_empty + NSV;  // [2]
  uint64_t* dp_full = s_full + 2;
  uint64_t* dp_free = s_full + 3;
  uint64_t* ds_ready = s_full + 4;
  uint64_t* dq_final = s_full + 5;
  uint64_t* drain = s_full + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h = blockIdx.y;
  const int qb = p.n_blk - 1 - blockIdx.x;  // deepest (usually heaviest) query blocks first
  const int g = h / (p.hq / p.hkv);
  const int32_t* rp = p.q_ptr + b * (p.n_blk + 1);
  const int e0 = rp[qb];
  const int n_it = rp[qb + 1] - e0;
  const int32_t* list = p.q_idx + int64_t(b) * p.cap + e0;
  const int row0 = b * p.t_pad + qb * kB;
  constexpr uint32_t T_S0 = 0, T_DP = 256, T_DQ = 384;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < NSK; ++s) {
      tc::mbar_init(k_full + s, 1);
      tc::mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < NSV; ++s) {
      tc::mbar_init(v_full + s, 1);
      tc::mbar_init(v_empty + s, 1);
    }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(s_full + 1, 1);
    tc::mbar_init(dp_full, 1);
    tc::mbar_init(dp_free, 128 * kNWG);
    tc::mbar_init(ds_ready, 128 * kNWG);
    tc::mbar_init(dq_final, 1);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kWMma) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWTma) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_it > 0) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      tc::tma_prefetch_desc(&tm_do);
      tc::mbar_arrive_expect_tx(q_full, 2 * TILE);
      for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sQ + c * kChunk, &tm_q, q_full, c * 64, h, row0);
      for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sDO + c * kChunk, &tm_do, q_full, c * 64, h, row0);
      // Use order: K(0), K(1), V(0), K(2), V(1), ...: K runs ahead of V.
      int kj = 0, vj = 0;
      bool ok = true;
      while (ok && (kj < n_it || vj < n_it)) {
        const bool do_k = kj < n_it && kj <= vj + 1;
        const int jj = do_k ? kj : vj;
        const int krow = b * p.t_pad + (list[jj] >> 1) * kB;
        if (do_k) {
          const int s = jj % NSK;
          if (!(ok = tc::mbar_wait(k_empty + s, ((jj / NSK) & 1) ^ 1, abort_flag, &g_status_bwd))) break;
          tc::mbar_arrive_expect_tx(k_full + s, TILE);
          for (int c = 0; c < NCH; ++c)
            tc::tma_load_3d(sK + s * TILE + c * kChunk, &tm_k, k_full + s, c * 64, g, krow);
          ++kj;
        } else {
          const int s = jj % NSV;
          if (!(ok = tc::mbar_wait(v_empty + s, ((jj / NSV) & 1) ^ 1, abort_flag, &g_status_bwd))) break;
          tc::mbar_arrive_expect_tx(v_full + s, TILE);
          for (int c = 0; c < NCH; ++c)
            tc::tma_load_3d(sV + s * TILE + c * kChunk, &tm_v, v_full + s, c * 64, g, krow);
          ++vj;
        }
      }
      if (*abort_flag) {
        volatile int never = 0;
        for (int jj = (kj > NSK ? kj - NSK : 0); jj < kj; ++jj)
          tc::mbar_wait(k_full + (jj % NSK), (jj / NSK) & 1, &never, &g_status_bwd, 100000000ull);
        for (int jj = (vj > NSV ? vj - NSV : 0); jj < vj; ++jj)
          tc::mbar_wait(v_full + (jj % NSV), (jj / NSV) & 1, &never, &g_status_bwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kWMma) {
    // ------------------------------------------------------------ MMA issuer
    // Per key tile j: dP(j+1) as soon as dP(j) has been read, dQ(j) once dS(j)
    // is in TMEM, then S(j+2) into the buffer dS(j) came from.
    if (lane == 0 && n_it > 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_q = tc::idesc_bf16(128, D, false, true);
      const uint32_t aQ = tc::smem_u32(sQ), aDO = tc::smem_u32(sDO), aK = tc::smem_u32(sK),
                     aV = tc::smem_u32(sV);
      auto issue_s = [&](int jj) -> bool {  // S(jj) = Q K^T into buffer jj % 2
        const int s = jj % NSK;
        if (!tc::mbar_wait(k_full + s, (jj / NSK) & 1, abort_flag, &g_status_bwd)) return false;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          tc::mma_ss(tmem + T_S0 + (jj & 1) * 128, tc::smem_desc(aQ + off, 16, 1024),
                     tc::smem_desc(aK + s * TILE + off, 16, 1024), idesc_s, k > 0);
        }
        tc::mma_commit(s_full + (jj & 1));
        return true;
      };
      auto issue_dp = [&](int jj) -> bool {  // dP(jj) = dO V^T
        const int s = jj % NSV;
        if (!tc::mbar_wait(v_full + s, (jj / NSV) & 1, abort_flag, &g_status_bwd)) return false;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          tc::mma_ss(tmem + T_DP, tc::smem_desc(aDO + off, 16, 1024),
                     tc::smem_desc(aV + s * TILE + off, 16, 1024), idesc_s, k > 0);
        }
        tc::mma_commit(dp_full);
        tc::mma_commit(v_empty + s);
        return true;
      };
      bool ok = tc::mbar_wait(q_full, 0, abort_flag, &g_status_bwd);
      ok = ok && issue_s(0);
      if (ok && n_it > 1) ok = issue_s(1);
      ok = ok && issue_dp(0);
      for (int jj = 0; ok && jj < n_it; ++jj) {
        if (jj + 1 < n_it) {
          if (!(ok = tc::mbar_wait(dp_free, jj & 1, abort_flag, &g_status_bwd))) break;
          if (!(ok = issue_dp(jj + 1))) break;
        }
        if (!(ok = tc::mbar_wait(ds_ready, jj & 1, abort_flag, &g_status_bwd))) break;
        tc::tc_fence_after();
        const int s = jj % NSK;
#pragma unroll
        for (int k = 0; k < kB / 16; ++k)  // dQ += dS K, dS packed bf16 in S buffer jj % 2
          mma_ts(tmem + T_DQ, wg_a(tmem + T_S0 + (jj & 1) * 128, k, 0),
                 tc::smem_desc(aK + s * TILE + k * 2048, kChunk, 1024), idesc_q, (jj > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(k_empty + s);
        if (jj + 2 < n_it && !(ok = issue_s(jj + 2))) break;  // buffer jj % 2: dS(jj) read above
      }
      if (ok) tc::mma_commit(dq_final);
      if (*abort_flag) {
        volatile int never = 0;
        tc::mma_commit(drain);
        tc::mbar_wait(drain, 0, &never, &g_status_bwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp < 4 * kNWG) {
    // ------------------------------------------------------------ compute warpgroups
    const int w = warp >> 2;          // key columns [32w, 32w+32) of this warpgroup
    const int r = threadIdx.x & 127;  // query row = TMEM lane
    const int i = qb * kB + r;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    constexpr int ESZ = F32OUT ? 4 : 2;
    constexpr int DW = D / kNWG;
    uint8_t* dq_row = static_cast<uint8_t*>(p.dq) + ((int64_t(row0 + r) * p.hq + h) * D + w * DW) * ESZ;
    auto wait_all = [&](uint64_t* b_, uint32_t par) {
      return __all_sync(0xffffffffu, tc::mbar_wait(b_, par, abort_flag, &g_status_bwd));
    };
    if (n_it == 0) {
      const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < DW * ESZ / 16; ++c) reinterpret_cast<uint4*>(dq_row)[c] = z;
    } else {
      const int64_t vec = (int64_t(b) * p.hq + h) * p.t_pad + i;
      const float nlse2 = -p.lse[vec] * kLog2e;
      const float drow = p.dvec[vec];
      const uint32_t* qmask_row = reinterpret_cast<const uint32_t*>(p.qmask + (int64_t(b) * p.cap + e0) * kB + r) + w;
      bool ok = true;
      int entry = list[0];
      uint32_t mk = (entry & 1) ? 0u : qmask_row[0];
      for (int jj = 0; jj < n_it; ++jj) {
        const bool full = entry & 1;
        const uint32_t mcur = mk;  // this group's 32 key columns
        if (jj + 1 < n_it) {
          entry = list[jj + 1];
          if (!(entry & 1)) mk = qmask_row[int64_t(jj + 1) * kB * 4];
        }
        const uint32_t tS = tmem + lane_base + T_S0 + (jj & 1) * 128;
        if (!wait_all(s_full + (jj & 1), (jj >> 1) & 1)) { ok = false; break; }
        tc::tc_fence_after();
        float pf[kCW];
        {
          uint32_t sv[kCW];
          tc::tmem_ld32(tS + kCW * w, sv);
          tc::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kCW; ++c) pf[c] = tc::ex2(fmaf(__uint_as_float(sv[c]), p.scale_log2, nlse2));
          if (!full) {
#pragma unroll
            for (int c = 0; c < kCW; ++c)
              if (!((mcur >> c) & 1u)) pf[c] = 0.f;
          }
        }
        if (!wait_all(dp_full, jj & 1)) { ok = false; break; }
        tc::tc_fence_after();
        {
          uint32_t dpv[kCW];
          tc::tmem_ld32(tmem + lane_base + T_DP + kCW * w, dpv);
          tc::tmem_ld_wait();
          tc::tc_fence_before();
          tc::mbar_arrive(dp_free);  // the dP region may be overwritten now
          uint32_t dw[kCW / 2];
#pragma unroll
          for (int u = 0; u < kCW / 2; ++u)
            dw[u] = tc::pack_bf16(pf[2 * u] * (__uint_as_float(dpv[2 * u]) - drow),
                                  pf[2 * u + 1] * (__uint_as_float(dpv[2 * u + 1]) - drow));
          tc::tmem_st16(tS + kCW * w, dw);  // dS over the first half of this group's S columns
          tc::tmem_st_wait();
        }
        tc::tc_fence_before();
        tc::mbar_arrive(ds_ready);
      }
      if (ok && wait_all(dq_final, 0)) {
        tc::tc_fence_after();
#pragma unroll
        for (int c = 0; c < DW / 16; ++c) {
          uint32_t v[16];
          tc::tmem_ld16(tmem + lane_base + T_DQ + w * DW + c * 16, v);
          tc::tmem_ld_wait();
          store_row16<F32OUT>(dq_row + c * 16 * ESZ, v, p.scale);
        }
      }
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kWMma) tc::tmem_dealloc(tmem, 512);
}

// D[b, h, i] = sum_d dO * O (fp32) for real rows, 0 for pad rows; one warp per
// (b, i, h) row.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                      const __nv_bfloat16* __restrict__ dout,
                                                      const int32_t* __restrict__ n_tokens, int32_t t_pad,
                                                      int32_t hq, int64_t n_rows, float* __restrict__ dvec) {
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
  float* dvec = static_cast<float*>(ws);  // workspace: D [B, Hq, T] fp32
  const int64_t n_rows = rows * hq;
  bwd_pre_kernel<D><<<grid_for(n_rows * 32, 256), 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), tree->n_tokens,
      tree->t_pad, hq, n_rows, dvec);
  TPA_CUDA_TRY(cudaGetLastError());

  CUtensorMap tq, tk, tv, tdo;
  if (!tmap::make_rows_heads_d(&tq, q, rows, hq, D) || !tmap::make_rows_heads_d(&tk, k, rows, hkv, D) ||
      !tmap::make_rows_heads_d(&tv, v, rows, hkv, D) || !tmap::make_rows_heads_d(&tdo, dout, rows, hq, D))
    return TPA_ERR_CUDA;
  BwdParams prm;
  prm.lse = lse;
  prm.dvec = dvec;
  prm.dq = dq;
  prm.dk = dk;
  prm.dv = dv;
  prm.subtree_end = tree->subtree_end;
  prm.n_tokens = tree->n_tokens;
  prm.k_ptr = mask->k_ptr;
  prm.k_idx = mask->k_idx;
  prm.q_ptr = mask->q_ptr;
  prm.q_idx = mask->q_idx;
  prm.qmask = reinterpret_cast<const uint4*>(mask->qmask);
  prm.t_pad = tree->t_pad;
  prm.n_blk = mask->n_blk;
  prm.cap = mask->cap;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.scale = scale;
  prm.scale_log2 = scale * kLog2e;
  TPA_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_kv_kernel<D, F32OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    KvCfg<D>::BYTES));
  attn_bwd_kv_kernel<D, F32OUT><<<dim3(mask->n_blk, hkv, tree->n_trees), kThreads, KvCfg<D>::BYTES, st>>>(
      tq, tk, tv, tdo, prm);
  TPA_CUDA_TRY(cudaGetLastError());
  TPA_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_dq_kernel<D, F32OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    DqCfg<D>::BYTES));
  attn_bwd_dq_kernel<D, F32OUT><<<dim3(mask->n_blk, hq, tree->n_trees), kThreads, DqCfg<D>::BYTES, st>>>(
      tq, tk, tv, tdo, prm);
  TPA_CUDA_TRY(cudaGetLastError());
  return TPA_OK;
}

}  // namespace

TPA_DEFINE_STATUS_READER(tpa_internal_status_bwd, g_status_bwd)

extern "C" uint64_t tpa_tree_attn_bwd_workspace_bytes(int32_t n_trees, int32_t t_pad, int32_t n_heads_q,
                                                      int32_t head_dim, int32_t grad_dtype) {
  if (n_trees < 1 || t_pad < 1 || n_heads_q < 1 || head_dim < 1) return 0;
  if (grad_dtype != TPA_GRAD_F32 && grad_dtype != TPA_GRAD_BF16) return 0;
  return align256(uint64_t(n_trees) * uint64_t(t_pad) * uint64_t(n_heads_q) * 4);
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
// them the backward's scratch (D = rowsum(dO * O)) lives in one fixed array
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
