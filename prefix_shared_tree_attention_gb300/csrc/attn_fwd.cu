// Tree attention forward on tcgen05 tensor cores (sm_103a).
//
// Semantics (tree training page, §树构建过程 mask caption, §注意力机制): query
// i of a packed tree sees key j iff j <= i <= E[j] (j is i or an ancestor);
// O_i = softmax over the visible keys of scale * q_i.k_j, times v_j.
// Only non-empty 128x128 tiles are visited (the per-query-block CSR of the
// classifier); PARTIAL tiles apply the precomputed 128-bit row masks, FULL
// tiles apply nothing.
//
// One CTA = one 128-query tile of NH query heads that share a key/value head
// (NH = 2 when the group size allows it), so every K/V tile is loaded once
// for both heads and the mask is shared.  Warp roles:
//   warpgroup h < NH  softmax of head h: thread r owns query row r (TMEM lane
//                     r); fp32 online softmax in the log2 domain with packed
//                     f32x2 arithmetic; P (bf16) goes to TMEM over the S
//                     columns it replaces and feeds the TS-form PV MMA;
//                     O is rescaled in TMEM only when the running max grows
//                     by more than 2^8 (exact: numerator and denominator keep
//                     the same stale max).
//   warp 4*NH         TMA producer: Q of each head once, then K and V tiles
//                     through separate rings.
//   warp 4*NH+1       MMA issuer (one thread).  Per key tile j and head h:
//                     PV_h(j) then S_h(j+1), so head B's softmax runs while
//                     head A's MMAs run (ping-pong) and the tensor core always
//                     has the other head's work queued.
// TMEM columns: S_h [128h, 128h+128) (P_h aliased on its first 64 columns),
// O_h [128 NH + 128h, ...).
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
constexpr uint32_t kSmemMax = 232448;      // 227 KB opt-in per CTA

struct FwdParams {
  __nv_bfloat16* o;
  float* lse;
  const int32_t* n_tokens;
  const int32_t* q_ptr;
  const int32_t* q_idx;
  const uint4* qmask;
  int32_t t_pad, n_blk, cap, hq, hkv;
  float scale_log2;  // softmax scale * log2(e)
};

template <int D, int NH>
struct FwdCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = NCH * kChunk;   // one 128 x D bf16 tile
  static constexpr uint32_t BASE = NH * TILE + 4096;
  static constexpr int NS_FIT = int((kSmemMax - 1024 - BASE) / (2 * TILE));
  static constexpr int NS = NS_FIT > 3 ? 3 : NS_FIT;  // K and V ring depth
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NH * TILE;
  static constexpr uint32_t OFF_V = OFF_K + NS * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + NS * TILE;
  // q_full, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[NH], p_full[NH], o_final, drain
  static constexpr int NBAR = 1 + 4 * NS + 2 * NH + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 16 + 1024;  // + alignment slack
  static constexpr int THREADS = 128 * NH + 64;
  static constexpr uint32_t TMEM_COLS = NH == 2 ? 512 : 256;
  static_assert(NS >= 1, "shared memory too small");
  static_assert(BYTES <= kSmemMax, "shared memory budget");
};

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// O_h (+)= P_h V with P_h read from TMEM (TS form of tcgen05.mma).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  tc::tmem_st32(taddr, *reinterpret_cast<const uint32_t(*)[32]>(r));
  tc::tmem_st32(taddr + 32, *reinterpret_cast<const uint32_t(*)[32]>(r + 32));
}

template <int D, int NH>
__global__ void __launch_bounds__(FwdCfg<D, NH>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using C = FwdCfg<D, NH>;
  constexpr int NCH = C::NCH, NS = C::NS;
  constexpr uint32_t TILE = C::TILE;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bar;
  uint64_t* k_full = bar + 1;
  uint64_t* k_empty = bar + 1 + NS;
  uint64_t* v_full = bar + 1 + 2 * NS;
  uint64_t* v_empty = bar + 1 + 3 * NS;
  uint64_t* s_full = bar + 1 + 4 * NS;
  uint64_t* p_full = bar + 1 + 4 * NS + NH;
  uint64_t* o_final = bar + 1 + 4 * NS + 2 * NH;
  uint64_t* drain = o_final + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z;
  const int h0 = blockIdx.y * NH;  // first query head of this CTA
  const int qb = p.n_blk - 1 - blockIdx.x;  // deepest (usually heaviest) query blocks first
  const int g = h0 / (p.hq / p.hkv);
  const int32_t* rp = p.q_ptr + b * (p.n_blk + 1);
  const int e0 = rp[qb];
  const int n_it = rp[qb + 1] - e0;
  const int32_t* list = p.q_idx + int64_t(b) * p.cap + e0;
  const int row0 = b * p.t_pad + qb * kB;  // global row of the tile's first query
  constexpr int W_TMA = 4 * NH, W_MMA = 4 * NH + 1;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(k_full + s, 1);
      tc::mbar_init(k_empty + s, 1);
      tc::mbar_init(v_full + s, 1);
      tc::mbar_init(v_empty + s, 1);
    }
    for (int h = 0; h < NH; ++h) {
      tc::mbar_init(s_full + h, 1);
      tc::mbar_init(p_full + h, 128);
    }
    tc::mbar_init(o_final, 1);
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == W_MMA) tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == W_TMA) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_it > 0) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      tc::mbar_arrive_expect_tx(q_full, NH * TILE);
      for (int h = 0; h < NH; ++h)
        for (int c = 0; c < NCH; ++c)
          tc::tma_load_3d(sQ + h * TILE + c * kChunk, &tm_q, q_full, c * 64, h0 + h, row0);
      // K runs ahead of V by one tile: the MMA needs K(j+1) before V(j).
      int kj = 0, vj = 0;
      bool ok = true;
      while (ok && (kj < n_it || vj < n_it)) {
        const bool do_k = kj < n_it && kj <= vj + 1;
        const int j = do_k ? kj : vj;
        const int s = j % NS;
        const int krow = b * p.t_pad + (list[j] >> 1) * kB;
        if (do_k) {
          if (!(ok = tc::mbar_wait(k_empty + s, ((j / NS) & 1) ^ 1, abort_flag, &g_status_fwd))) break;
          tc::mbar_arrive_expect_tx(k_full + s, TILE);
          for (int c = 0; c < NCH; ++c)
            tc::tma_load_3d(sK + s * TILE + c * kChunk, &tm_k, k_full + s, c * 64, g, krow);
          ++kj;
        } else {
          if (!(ok = tc::mbar_wait(v_empty + s, ((j / NS) & 1) ^ 1, abort_flag, &g_status_fwd))) break;
          tc::mbar_arrive_expect_tx(v_full + s, TILE);
          for (int c = 0; c < NCH; ++c)
            tc::tma_load_3d(sV + s * TILE + c * kChunk, &tm_v, v_full + s, c * 64, g, krow);
          ++vj;
        }
      }
      if (*abort_flag) {  // let the copies already issued land before the CTA exits
        volatile int never = 0;
        for (int j = (kj > NS ? kj - NS : 0); j < kj; ++j)
          tc::mbar_wait(k_full + (j % NS), (j / NS) & 1, &never, &g_status_fwd, 100000000ull);
        for (int j = (vj > NS ? vj - NS : 0); j < vj; ++j)
          tc::mbar_wait(v_full + (j % NS), (j / NS) & 1, &never, &g_status_fwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_it > 0) {
      constexpr uint32_t idesc_qk = tc::idesc_bf16(128, 128, false, false);
      constexpr uint32_t idesc_pv = tc::idesc_bf16(128, D, false, true);
      const uint32_t aQ = tc::smem_u32(sQ), aK = tc::smem_u32(sK), aV = tc::smem_u32(sV);
      auto issue_s = [&](int h, int s) {  // S_h = Q_h K(s)^T
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off = (k >> 2) * kChunk + (k & 3) * 32;
          tc::mma_ss(tmem + h * 128, tc::smem_desc(aQ + h * TILE + off, 16, 1024),
                     tc::smem_desc(aK + s * TILE + off, 16, 1024), idesc_qk, k > 0);
        }
      };
      auto issue_pv = [&](int h, int s, bool first) {  // O_h (+)= P_h V(s), P_h read from TMEM
#pragma unroll
        for (int k = 0; k < kB / 16; ++k) {
          const uint64_t db = tc::smem_desc(aV + s * TILE + k * 2048, kChunk, 1024);
          mma_ts(tmem + 128 * NH + h * 128, tmem + h * 128 + k * 8, db, idesc_pv, (!first || k > 0) ? 1u : 0u);
        }
      };
      bool ok = tc::mbar_wait(q_full, 0, abort_flag, &g_status_fwd) &&
                tc::mbar_wait(k_full, 0, abort_flag, &g_status_fwd);
      if (ok) {
        tc::tc_fence_after();
        for (int h = 0; h < NH; ++h) {
          issue_s(h, 0);
          tc::mma_commit(s_full + h);
        }
        tc::mma_commit(k_empty);
      }
      for (int j = 0; ok && j < n_it; ++j) {
        const int s = j % NS, s1 = (j + 1) % NS;
        const bool more = j + 1 < n_it;
        if (!(ok = tc::mbar_wait(v_full + s, (j / NS) & 1, abort_flag, &g_status_fwd))) break;
        for (int h = 0; h < NH && ok; ++h) {
          if (!(ok = tc::mbar_wait(p_full + h, j & 1, abort_flag, &g_status_fwd))) break;
          tc::tc_fence_after();
          issue_pv(h, s, j == 0);
          if (more) {
            if (h == 0 && !(ok = tc::mbar_wait(k_full + s1, ((j + 1) / NS) & 1, abort_flag, &g_status_fwd)))
              break;
            tc::tc_fence_after();
            issue_s(h, s1);
            tc::mma_commit(s_full + h);
          }
        }
        if (!ok) break;
        tc::mma_commit(v_empty + s);
        if (more) tc::mma_commit(k_empty + s1);
      }
      if (ok) tc::mma_commit(o_final);
      if (*abort_flag) {  // let issued MMAs finish before TMEM is released
        volatile int never = 0;
        tc::mma_commit(drain);
        tc::mbar_wait(drain, 0, &never, &g_status_fwd, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (head h)
    const int h = warp >> 2;
    const int r = threadIdx.x & 127;   // query row within the tile = TMEM lane
    const int i = qb * kB + r;         // query position in the tree
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + h * 128;
    const uint32_t tO = tmem + lane_base + 128 * NH + h * 128;
    __nv_bfloat16* orow = p.o + (int64_t(row0 + r) * p.hq + h0 + h) * D;
    float* lse_out = p.lse + (int64_t(b) * p.hq + h0 + h) * p.t_pad + i;
    auto wait_all = [&](uint64_t* b_, uint32_t par) {
      return __all_sync(0xffffffffu, tc::mbar_wait(b_, par, abort_flag, &g_status_fwd));
    };
    if (n_it == 0) {
      const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
      *lse_out = 0.f;
    } else {
      const uint64_t sl2 = f2(p.scale_log2, p.scale_log2);
      const uint4* qmask_row = p.qmask + (int64_t(b) * p.cap + e0) * kB + r;
      float m_run = -INFINITY, l_run = 0.f;
      bool ok = true;
      int entry = list[0];
      uint4 mk = (entry & 1) ? make_uint4(0, 0, 0, 0) : qmask_row[0];
      for (int j = 0; j < n_it; ++j) {
        const bool full = entry & 1;
        const uint4 mcur = mk;
        if (j + 1 < n_it) {  // prefetch the next tile's entry and mask row
          entry = list[j + 1];
          if (!(entry & 1)) mk = qmask_row[int64_t(j + 1) * kB];
        }
        if (!wait_all(s_full + h, j & 1)) { ok = false; break; }
        tc::tc_fence_after();
        uint32_t sv[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tc::tmem_ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sv + c * 32));
        tc::tmem_ld_wait();
        if (!full) {
          const uint32_t w[4] = {mcur.x, mcur.y, mcur.z, mcur.w};
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (!((w[c >> 5] >> (c & 31)) & 1u)) sv[c] = 0xff800000u;  // -inf
        }
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 128; c += 2) mx = max3(mx, __uint_as_float(sv[c]), __uint_as_float(sv[c + 1]));
        const float m_new = fmaxf(m_run, mx * p.scale_log2);
        const bool resc = m_new > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
          alpha = tc::ex2(m_run - m_new);
          m_run = m_new;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        const uint64_t negm = f2(-m_use, -m_use);
        uint64_t sum2 = f2(0.f, 0.f);
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float a, bb;
          unf2(fma2(f2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), sl2, negm), a, bb);
          const float p0 = tc::ex2(a), p1 = tc::ex2(bb);
          sum2 = add2(sum2, f2(p0, p1));
          pk[c] = tc::pack_bf16(p0, p1);
        }
        float s_lo, s_hi;
        unf2(sum2, s_lo, s_hi);
        l_run = l_run * alpha + (s_lo + s_hi);

        // O_h holds the result of PV_h(j-1): s_full(j) was committed after it.
        if (j >= 1 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            tc::tmem_ld32(tO + c * 32, ov);
            tc::tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 32; ++u) ov[u] = __float_as_uint(__uint_as_float(ov[u]) * alpha);
            tc::tmem_st32(tO + c * 32, ov);
          }
        }
        tmem_st64(tS, pk);  // P over the first 64 columns of S (packed bf16 pairs)
        tc::tmem_st_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(p_full + h);
      }
      if (ok && wait_all(o_final, 0)) {
        tc::tc_fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t ov[32];
          tc::tmem_ld32(tO + c * 32, ov);
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
  if (warp == W_MMA) tc::tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, int NH>
int launch_fwd_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& prm,
                   int n_blk, int hq, int n_trees, cudaStream_t st) {
  using C = FwdCfg<D, NH>;
  TPA_CUDA_TRY(cudaFuncSetAttribute(attn_fwd_kernel<D, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES));
  attn_fwd_kernel<D, NH><<<dim3(n_blk, hq / NH, n_trees), C::THREADS, C::BYTES, st>>>(tq, tk, tv, prm);
  TPA_CUDA_TRY(cudaGetLastError());
  return TPA_OK;
}

template <int D>
int launch_fwd(const tpa_tree_view* tree, const tpa_blockmask_view* mask, const void* q, const void* k,
               const void* v, void* o, float* lse, int hq, int hkv, float scale, cudaStream_t st) {
  const uint64_t rows = uint64_t(tree->n_trees) * tree->t_pad;
  CUtensorMap tq, tk, tv;
  if (!tmap::make_rows_heads_d(&tq, q, rows, hq, D) || !tmap::make_rows_heads_d(&tk, k, rows, hkv, D) ||
      !tmap::make_rows_heads_d(&tv, v, rows, hkv, D))
    return TPA_ERR_CUDA;
  FwdParams prm;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.n_tokens = tree->n_tokens;
  prm.q_ptr = mask->q_ptr;
  prm.q_idx = mask->q_idx;
  prm.qmask = reinterpret_cast<const uint4*>(mask->qmask);
  prm.t_pad = tree->t_pad;
  prm.n_blk = mask->n_blk;
  prm.cap = mask->cap;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.scale_log2 = scale * kLog2e;
  if ((hq / hkv) % 2 == 0) return launch_fwd_cfg<D, 2>(tq, tk, tv, prm, mask->n_blk, hq, tree->n_trees, st);
  return launch_fwd_cfg<D, 1>(tq, tk, tv, prm, mask->n_blk, hq, tree->n_trees, st);
}

}  // namespace

TPA_DEFINE_STATUS_READER(tpa_internal_status_fwd, g_status_fwd)

int tpa_internal_check_attn_args(const tpa_tree_view* tree, const tpa_blockmask_view* mask, int hq,
                                 int hkv, int d) {
  if (!tree || !mask || !tree->subtree_end || !tree->n_tokens || !mask->q_ptr || !mask->q_idx ||
      !mask->k_ptr || !mask->k_idx || !mask->qmask)
    return TPA_ERR_INVALID_ARG;
  if (tree->n_trees < 1 || tree->n_trees > 65535 || tree->t_pad < kB || tree->t_pad % kB ||
      mask->n_trees != tree->n_trees || mask->n_blk != tree->t_pad / kB)
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
