// Tree attention backward on tcgen05 tensor cores (sm_103a).
//
// Gradients of <dO, O> for the tree attention forward (tree training page,
// §树构建过程 mask caption: query i sees key j iff j <= i <= E[j]):
//   P_ij = exp(scale q_i.k_j - LSE_i),   D_i = dO_i . O_i
//   dV_j = sum_i P_ij dO_i,   dS_ij = P_ij (dO_i . v_j - D_i)
//   dQ_i = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i
// with dK/dV summed over the query heads of each key/value head.
//
// Three kernels, no atomics on the hot loop:
//  (1) preprocess: D = rowsum(dO * O) in fp32 (and zeroed fp32 rows of the
//      key tiles whose long column is split into several items that add into
//      them: the dK/dV outputs for fp32 gradients, staging rows for bf16
//      gradients, whose last adder converts them to bf16).
//  (2) KV kernel: work items are (key tile, kv head, tree, chunk of that key
//      tile's column, sized from the tree's ancestor pairs so that the items
//      balance over the SMs), a step being one (query head, query tile) pair
//      of the per-key-block CSR.  Per step the MMA issuer runs
//      S^T = K Q^T and dP^T = V dO^T into two TMEM regions that swap roles
//      every step; four compute warpgroups (thread r = key row r = TMEM lane
//      r; warpgroup w = query columns [32w, 32w+32)) write P^T and dS^T back
//      into the S^T region as packed bf16, and the issuer runs dV += P^T dO
//      and dK += dS^T Q with A read from TMEM, issuing the next step's S^T as
//      soon as this step's dP^T has been read.  A key only sees the query
//      interval [j, E[j]], applied on PARTIAL tiles.
//  (3) dQ kernel: work items are (query tile, query head, tree); it walks the
//      query block's key tiles like the forward, rotating S, dP and packed dS
//      through three TMEM regions so the next tile's S and dP run while this
//      tile's dS is formed: dS = P (dP - D) with the forward's LSE and the
//      partial-tile bit masks, dQ += dS K accumulated in TMEM; dQ is stored
//      once.  With d = 128 and an even number of query heads per key/value
//      head, the pair form of this kernel runs two heads of a group on the
//      two SMs of a TPC with M = 256 MMAs (cta_group::2), each SM holding
//      half of every B operand.
// Both main kernels are persistent: one CTA per SM takes items from a counter
// in the block-mask buffer and barrier phases run on across items.  The TMA
// producer and MMA issuer warps run their whole loops on one elected thread:
// a warp-level sync right after tcgen05.mma holds the warp until the queued
// MMAs have entered the tensor pipe, which would leave the pipe idle for the
// length of every wait between MMA groups.
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
constexpr uint32_t kChunk = 128 * 128;    // bytes of a 128-row x 64-col bf16 tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kSmemMax = 232448;   // 227 KB opt-in per CTA
constexpr int kNWG = 4;                    // compute warpgroups per CTA
constexpr int kThreads = 128 * kNWG + 64;  // + TMA warp + MMA warp
constexpr int kWTma = 4 * kNWG, kWMma = 4 * kNWG + 1;
constexpr int kCW = kB / kNWG;             // query or key columns per warpgroup (32)
constexpr int kKvChunkMin = 64;            // fewest steps per KV work item of a split column

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
  uint32_t* sched;      // work counters: [2..3] KV kernel, [4..5] dQ kernel
  float* stage_k;       // bf16 gradients: fp32 dK, dV rows of split key columns [B, T, Hkv, d]
  float* stage_v;
  uint32_t* kv_cnt;     // bf16 gradients: finished items per (tree, kv head, key tile, compute warp)
  int32_t t_pad, n_blk, cap, hq, hkv;
  int32_t n_trees, kv_chunk, kv_nchunk, kv_items, dq_items;
  int32_t wide;  // gradient outputs 32-byte aligned: rows stored 32 bytes (one sector) at a time
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

__device__ __forceinline__ void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}

__device__ __forceinline__ void st_v8(void* addr, const uint32_t (&v)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(addr), "r"(v[0]), "r"(v[1]),
               "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
               : "memory");
}

// Writes 16 fp32 values of one row as fp32 or bf16 (with a scale), or adds
// them into an fp32 row.  `wide`: the row is 32-byte aligned and goes out in
// 32-byte stores (one full sector each: two for fp32, one for bf16) instead
// of 16-byte ones.
template <bool F32OUT>
__device__ __forceinline__ void store_row16(uint8_t* dst, const uint32_t (&v)[16], float scale, bool add,
                                            bool wide = false) {
  if (F32OUT) {
    float* f = reinterpret_cast<float*>(dst);
    if (!add && wide) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = __float_as_uint(__uint_as_float(v[8 * h + e]) * scale);
        st_v8(f + 8 * h, w);
      }
      return;
    }
    if (add) {
#pragma unroll
      for (int t = 0; t < 4; ++t)
        red_add_v4(f + 4 * t, __uint_as_float(v[4 * t]) * scale, __uint_as_float(v[4 * t + 1]) * scale,
                   __uint_as_float(v[4 * t + 2]) * scale, __uint_as_float(v[4 * t + 3]) * scale);
    } else {
      uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
      for (int t = 0; t < 4; ++t)
        d4[t] = make_uint4(__float_as_uint(__uint_as_float(v[4 * t]) * scale),
                           __float_as_uint(__uint_as_float(v[4 * t + 1]) * scale),
                           __float_as_uint(__uint_as_float(v[4 * t + 2]) * scale),
                           __float_as_uint(__uint_as_float(v[4 * t + 3]) * scale));
    }
  } else {
    uint32_t w[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      w[u] = tc::pack_bf16(__uint_as_float(v[2 * u]) * scale, __uint_as_float(v[2 * u + 1]) * scale);
    if (wide) {  // one full 32-byte sector per store
      st_v8(dst, w);
      return;
    }
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// The last CTA to finish rearms a kernel's work counter for the next call.
__device__ __forceinline__ void rearm_counter(uint32_t* ctr) {
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(ctr + 1, 1u) == gridDim.x - 1) {
      ctr[0] = 0;
      ctr[1] = 0;
      __threadfence();
    }
  }
}

// =========================================================================== KV kernel
//
// A step is one (query head, 128-query tile) pair of a key tile's column.
// TMEM: two 128-column regions X = [0, 128) and Y = [128, 256) and the dV, dK
// accumulators in [256, 256+D) and [256+D, 256+2D).  Step t computes S^T(t)
// into region A_t and dP^T(t) into the other region B_t, alternating with t
// (A_t = X for even t).  Compute warpgroup w owns query columns [32w, 32w+32)
// of both; it writes P^T(t) packed into the first 16 of its S^T columns and
// dS^T(t) packed into the other 16, so B_t is free as soon as dP^T(t) has
// been read.  The issuer then runs S^T(t+1) into B_t (= A_{t+1}) while dV(t)
// and dK(t) read A_t, and dP^T(t+1) into A_t (= B_{t+1}) behind them.

template <int D>
struct KvCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = NCH * kChunk;  // 128-row tile of K, V, Q or dO
  // Q ring one stage deeper than the dO ring: Q(t) feeds S^T(t), which is
  // issued a step before dP^T(t), and dK(t), the step's last MMA.  LSE
  // travels with dO (read before P^T(t) is published, so the dO stage frees
  // once dV(t) is done), D with Q (read until dS^T(t) is published).
  static constexpr int NSQ = D == 128 ? 3 : 4;
  static constexpr int NSD = D == 128 ? 2 : 3;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + TILE;
  static constexpr uint32_t OFF_Q = OFF_V + TILE;
  static constexpr uint32_t OFF_DO = OFF_Q + NSQ * TILE;
  static constexpr uint32_t OFF_LSE = OFF_DO + NSD * TILE;    // NSD x 128 fp32
  static constexpr uint32_t OFF_DV = OFF_LSE + NSD * kB * 4;  // NSQ x 128 fp32
  static constexpr uint32_t OFF_BAR = OFF_DV + NSQ * kB * 4;
  // kv_full, kv_empty, q_full[NSQ], q_empty[NSQ], do_full[NSD], do_empty[NSD], s_full, dp_full,
  // p_ready, dp_free, ds_ready, acc_full, acc_free, drain, item_full[2], item_empty[2]
  static constexpr int NBAR = 2 + 2 * NSQ + 2 * NSD + 8 + 4;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  // No alignment slack: the kernel checks that dynamic shared memory starts
  // 1024-byte aligned (the swizzled tiles need it).
  static constexpr uint32_t BYTES = OFF_MISC + 32;
  static_assert(BYTES <= kSmemMax, "shared memory budget");
};

struct KvItem {
  int b, g, kb, n_col, s0, n;  // column of (b, g, kb); steps [s0, s0 + n)
  const int32_t* list;
};

__device__ __forceinline__ KvItem decode_kv(const BwdParams& p, int it) {
  KvItem r;
  const int G = p.hq / p.hkv;
  // (tree, kv head) slowest so the Q/dO tiles of one head group stay in L2
  // while its columns run; ascending key blocks (the longest columns first);
  // the chunk fastest.  Chunks past a column's end are empty and skipped by
  // the producer.
  const int per_g = p.n_blk * p.kv_nchunk;
  const int per_b = p.hkv * per_g;
  r.b = it / per_b;
  int rem = it - r.b * per_b;
  r.g = rem / per_g;
  rem -= r.g * per_g;
  r.kb = rem / p.kv_nchunk;
  const int ch = rem - r.kb * p.kv_nchunk;
  const int32_t* kp = p.k_ptr + r.b * (p.n_blk + 1);
  r.n_col = kp[r.kb + 1] - kp[r.kb];
  r.list = p.k_idx + int64_t(r.b) * p.cap + kp[r.kb];
  r.s0 = ch * p.kv_chunk;
  const int total = G * r.n_col;
  r.n = total - r.s0 < p.kv_chunk ? total - r.s0 : p.kv_chunk;
  return r;
}

// Descriptor offset (>> 4) of the 16-column K slice k of a swizzled tile
// whose 64-column chunks are `chunk` bytes apart (kChunk for 128 rows).
__device__ __forceinline__ uint32_t kslice(int k, uint32_t chunk = kChunk) {
  return ((k >> 2) * chunk + (k & 3) * 32) >> 4;
}

// TMEM column of the packed bf16 A operand for the 16-row K slice kk of a
// region whose warpgroup w wrote its 32 values packed into columns
// [32w + half, 32w + half + 16) (half = 0 for P, 16 for dS).
__device__ __forceinline__ uint32_t packed_a(uint32_t region, int half, int kk) {
  return region + 32 * (kk >> 1) + half + 8 * (kk & 1);
}

template <int D, bool F32OUT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using C = KvCfg<D>;
  constexpr int NCH = C::NCH, NSQ = C::NSQ, NSD = C::NSD;
  constexpr uint32_t TILE = C::TILE;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (tc::smem_u32(smem) & 1023u) {  // uniform over the CTA: every thread leaves
    if (threadIdx.x == 0) atomicOr(&g_status_bwd, 2u);
    return;
  }
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  float* sLSE = reinterpret_cast<float*>(smem + C::OFF_LSE);
  float* sDv = reinterpret_cast<float*>(smem + C::OFF_DV);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bar;
  uint64_t* kv_empty = bar + 1;
  uint64_t* q_full = bar + 2;
  uint64_t* q_empty = q_full + NSQ;
  uint64_t* do_full = q_empty + NSQ;
  uint64_t* do_empty = do_full + NSD;
  uint64_t* s_full = do_empty + NSD;
  uint64_t* dp_full = s_full + 1;
  uint64_t* p_ready = s_full + 2;
  uint64_t* dp_free = s_full + 3;
  uint64_t* ds_ready = s_full + 4;
  uint64_t* acc_full = s_full + 5;
  uint64_t* acc_free = s_full + 6;
  uint64_t* drain = s_full + 7;
  uint64_t* item_full = s_full + 8;   // [2]
  uint64_t* item_empty = s_full + 10;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* item_ring = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);  // [2]

  const int warp = threadIdx.x >> 5;
  const int G = p.hq / p.hkv;
  constexpr uint32_t T_DV = 256, T_DK = 256 + D;
  constexpr int NCONS = 1 + 4 * kNWG;  // item consumers: MMA warp (elected lane) + one per compute warp
  // region holding S^T of global step gs (dP^T goes to the other one)
  auto reg_s = [](int gs) -> uint32_t { return (gs & 1) ? 128u : 0u; };

  if (threadIdx.x == 0) {
    tc::mbar_init(kv_full, 1);
    tc::mbar_init(kv_empty, 1);
    for (int s = 0; s < NSQ; ++s) {
      tc::mbar_init(q_full + s, 1);
      tc::mbar_init(q_empty + s, 1);
    }
    for (int s = 0; s < NSD; ++s) {
      tc::mbar_init(do_full + s, 1);
      tc::mbar_init(do_empty + s, 1);
    }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(dp_full, 1);
    // compute-side barriers take one arrival per warp (after __syncwarp): 512
    // single-thread arrivals on one barrier word would queue up
    tc::mbar_init(p_ready, 4 * kNWG);
    tc::mbar_init(dp_free, 4 * kNWG);
    tc::mbar_init(ds_ready, 4 * kNWG);
    tc::mbar_init(acc_full, 1);
    tc::mbar_init(acc_free, 4 * kNWG);
    tc::mbar_init(drain, 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(item_full + s, 1);
      tc::mbar_init(item_empty + s, NCONS);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kWMma) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The dQ kernel after this one neither reads nor writes what this one
  // writes: it may take the SMs this kernel's CTAs leave.  It reads D, so
  // it is let go only once the preprocess before this kernel has completed.
  if (threadIdx.x == 0) {
    tc::grid_wait_prior();
    tc::grid_launch_dependents();
  }
  auto wait_u = [&](uint64_t* b_, uint32_t par) {
    return __all_sync(0xffffffffu, tc::mbar_wait(b_, par, abort_flag, &g_status_bwd));
  };
  // one arrival for the warp, after every lane's own fences and stores
  auto warp_arrive = [&](uint64_t* b_) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive(b_);
  };

  if (warp == kWTma) {
    // ------------------------------------------------------------ producer
    // One thread runs the whole loop, like the MMA issuer: a warp-level sync
    // right after the bulk copies would hold the warp until they are issued.
    if (tc::elect_one()) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      tc::tma_prefetch_desc(&tm_do);
      tc::grid_wait_prior();  // D, loaded with each Q stage, comes from the preprocess
      auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_bwd); };
      int qs = 0, nk = 0, nq_half = 0;  // steps loaded, K/V loads, and a lone Q load in flight
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (!(ok = wait1(item_empty + (k & 1), ((k >> 1) & 1) ^ 1))) break;
        // Take indices until one has work (bf16 outputs also need the zero
        // rows of key tiles no query sees); only that one is handed on.
        int it = -1;
        KvItem I;
        for (;;) {
          const uint32_t u = atomicAdd(p.sched + 2, 1u);
          if (u >= uint32_t(p.kv_items)) break;  // unsigned: no index below 0
          I = decode_kv(p, int(u));
          if (I.n > 0 || (!F32OUT && I.s0 == 0)) {
            it = int(u);
            break;
          }
        }
        item_ring[k & 1] = it;
        tc::mbar_arrive(item_full + (k & 1));
        if (it < 0) break;
        if (I.n <= 0) continue;
        const int krow = I.b * p.t_pad + I.kb * kB;
        if (!(ok = wait1(kv_empty, (nk & 1) ^ 1))) break;
        tc::mbar_arrive_expect_tx(kv_full, 2 * TILE);
        for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sK + c * kChunk, &tm_k, kv_full, c * 64, I.g, krow);
        for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sV + c * kChunk, &tm_v, kv_full, c * 64, I.g, krow);
        ++nk;
        int entry = I.list[I.s0 % I.n_col];
        for (int t = 0; t < I.n; ++t) {
          const int sq = qs % NSQ, sd = qs % NSD;
          const int s = I.s0 + t;
          const int h = I.g * G + s / I.n_col;
          const int qb = entry >> 1;
          if (t + 1 < I.n) entry = I.list[(s + 1) % I.n_col];
          const int qrow = I.b * p.t_pad + qb * kB;
          const int64_t vec = (int64_t(I.b) * p.hq + h) * p.t_pad + qb * kB;
          if (!(ok = wait1(q_empty + sq, ((qs / NSQ) & 1) ^ 1))) break;
          tc::mbar_arrive_expect_tx(q_full + sq, TILE + kB * 4);
          for (int c = 0; c < NCH; ++c)
            tc::tma_load_3d(sQ + sq * TILE + c * kChunk, &tm_q, q_full + sq, c * 64, h, qrow);
          tc::bulk_load(sDv + sq * kB, p.dvec + vec, kB * 4, q_full + sq);
          nq_half = 1;  // this step's Q load is in flight, its dO load not yet
          if (!(ok = wait1(do_empty + sd, ((qs / NSD) & 1) ^ 1))) break;
          tc::mbar_arrive_expect_tx(do_full + sd, TILE + kB * 4);
          for (int c = 0; c < NCH; ++c)
            tc::tma_load_3d(sDO + sd * TILE + c * kChunk, &tm_do, do_full + sd, c * 64, h, qrow);
          tc::bulk_load(sLSE + sd * kB, p.lse + vec, kB * 4, do_full + sd);
          nq_half = 0;
          ++qs;
        }
      }
      if (*abort_flag) {  // let the copies already issued land before the CTA exits
        volatile int never = 0;
        if (nk > 0) tc::mbar_wait(kv_full, (nk - 1) & 1, &never, &g_status_bwd, 100000000ull);
        const int nq = qs + nq_half;  // Q loads issued
        for (int j = (nq > NSQ ? nq - NSQ : 0); j < nq; ++j)
          tc::mbar_wait(q_full + (j % NSQ), (j / NSQ) & 1, &never, &g_status_bwd, 100000000ull);
        for (int j = (qs > NSD ? qs - NSD : 0); j < qs; ++j)
          tc::mbar_wait(do_full + (j % NSD), (j / NSD) & 1, &never, &g_status_bwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kWMma) {
    // ------------------------------------------------------------ MMA issuer
    // Per step t: dV(t) once P^T(t) is packed, S^T(t+1) into B_t once dP^T(t)
    // has been read, dK(t) once dS^T(t) is packed, then dP^T(t+1) into A_t
    // (in order behind dV(t) and dK(t), which read it).  One thread runs
    // the whole loop: a warp-level sync after tcgen05.mma holds the warp until
    // the thread's queued MMAs have gone into the pipe, so waits of a warp in
    // step would leave the tensor pipe idle between groups.
    constexpr uint32_t idesc_s = tc::idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_kv = tc::idesc_bf16(128, D, false, true);
    const uint64_t dK_ = tc::smem_desc(tc::smem_u32(sK), 16, 1024);
    const uint64_t dV_ = tc::smem_desc(tc::smem_u32(sV), 16, 1024);
    const uint64_t dQk = tc::smem_desc(tc::smem_u32(sQ), 16, 1024);        // Q as K-major B
    const uint64_t dDOk = tc::smem_desc(tc::smem_u32(sDO), 16, 1024);      // dO as K-major B
    const uint64_t dQm = tc::smem_desc(tc::smem_u32(sQ), kChunk, 1024);    // Q as MN-major B
    const uint64_t dDOm = tc::smem_desc(tc::smem_u32(sDO), kChunk, 1024);  // dO as MN-major B
    auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_bwd); };
    auto issue_s = [&](int gs) -> bool {  // S^T(gs) = K Q^T into A_gs
      if (!wait1(q_full + gs % NSQ, (gs / NSQ) & 1)) return false;
      tc::tc_fence_after();
      const uint32_t so = ((gs % NSQ) * TILE) >> 4;
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        tc::mma_ss(tmem + reg_s(gs), dK_ + kslice(k), dQk + so + kslice(k), idesc_s, k > 0);
      tc::mma_commit(s_full);
      return true;
    };
    auto issue_dp = [&](int gs) -> bool {  // dP^T(gs) = V dO^T into B_gs
      if (!wait1(do_full + gs % NSD, (gs / NSD) & 1)) return false;
      tc::tc_fence_after();
      const uint32_t so = ((gs % NSD) * TILE) >> 4;
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        tc::mma_ss(tmem + reg_s(gs + 1), dV_ + kslice(k), dDOk + so + kslice(k), idesc_s, k > 0);
      tc::mma_commit(dp_full);
      return true;
    };
    auto commit = [&](uint64_t* b_) { tc::mma_commit(b_); };
    if (tc::elect_one()) {
    int qs = 0, nk = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!(ok = wait1(item_full + (k & 1), (k >> 1) & 1))) break;
      const int it = item_ring[k & 1];
      tc::mbar_arrive(item_empty + (k & 1));
      if (it < 0) break;
      const KvItem I = decode_kv(p, it);
      const int n = I.n;
      if (n <= 0) continue;
      if (!(ok = wait1(kv_full, nk & 1))) break;
      tc::tc_fence_after();
      if (!(ok = issue_s(qs) && issue_dp(qs))) break;
      if (n == 1) commit(kv_empty);  // K and V are read by S^T and dP^T only
      for (int t = 0; ok && t < n; ++t) {
        const int gs = qs + t, sq = gs % NSQ, sd = gs % NSD;
        const uint32_t soq = (sq * TILE) >> 4, sod = (sd * TILE) >> 4;
        const uint32_t A = tmem + reg_s(gs);
        if (!(ok = wait1(p_ready, gs & 1))) break;
        if (t == 0 && nk > 0 && !(ok = wait1(acc_free, (nk - 1) & 1))) break;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kB / 16; ++kk)  // dV += P^T dO, P^T packed bf16 in A_t
          mma_ts(tmem + T_DV, packed_a(A, 0, kk), dDOm + sod + ((kk * 2048) >> 4), idesc_kv,
                 (t > 0 || kk > 0) ? 1u : 0u);
        // dO(t) was last read by dV(t), its LSE before P^T(t) was published:
        // the stage is free once the MMAs issued so far are
        tc::mma_commit(do_empty + sd);
        // dV(t) keeps the tensor pipe busy while dP^T(t) is read out of B_t
        if (t + 1 < n) {
          if (!(ok = wait1(dp_free, gs & 1))) break;
          if (!(ok = issue_s(gs + 1))) break;
        }
        if (!(ok = wait1(ds_ready, gs & 1))) break;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kB / 16; ++kk)  // dK += dS^T Q, dS^T packed bf16 in A_t
          mma_ts(tmem + T_DK, packed_a(A, 16, kk), dQm + soq + ((kk * 2048) >> 4), idesc_kv,
                 (t > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(q_empty + sq);  // Q(t) read by S^T(t) and dK(t), its D before dS^T(t)
        if (t + 1 < n) {
          if (!(ok = issue_dp(gs + 1))) break;
          if (t + 2 == n) commit(kv_empty);
        }
      }
      if (!ok) break;
      commit(acc_full);  // dK, dV complete
      qs += n;
      ++nk;
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
    const int w = warp >> 2;              // query columns [32w, 32w+32) of each step
    const int r = threadIdx.x & 127;      // key row = TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    constexpr int ESZ = F32OUT ? 4 : 2;
    constexpr int DW = D / kNWG;
    int qs = 0, nk = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!wait_u(item_full + (k & 1), (k >> 1) & 1)) break;
      const int it = item_ring[k & 1];
      warp_arrive(item_empty + (k & 1));
      if (it < 0) break;
      const KvItem I = decode_kv(p, it);
      const int krow = I.b * p.t_pad + I.kb * kB;
      const int64_t off = ((int64_t(krow + r) * p.hkv + I.g) * D + w * DW) * ESZ;
      uint8_t* dk_row = static_cast<uint8_t*>(p.dk) + off;
      uint8_t* dv_row = static_cast<uint8_t*>(p.dv) + off;
      if (I.n <= 0) {
        // a key tile no query sees: zero rows (the preprocess zeroed fp32 outputs)
        if (!F32OUT && I.s0 == 0) {
          tc::grid_wait_prior();
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int c = 0; c < DW * ESZ / 16; ++c) {
            reinterpret_cast<uint4*>(dk_row)[c] = z;
            reinterpret_cast<uint4*>(dv_row)[c] = z;
          }
        }
        continue;
      }
      const int j = I.kb * kB + r;  // key position owned by this thread
      const int n_tok = p.n_tokens[I.b];
      const int Ej = (j < n_tok) ? p.subtree_end[krow + r] : -1;
      int entry = I.list[I.s0 % I.n_col];
      for (int t = 0; t < I.n; ++t) {
        const int gs = qs + t, st = gs % NSD, sq = gs % NSQ;  // LSE sits in the dO stage, D in the Q stage
        const int qb = entry >> 1;
        const bool full = entry & 1;
        if (t + 1 < I.n) entry = I.list[(I.s0 + t + 1) % I.n_col];
        const uint32_t tA = tmem + lane_base + reg_s(gs) + kCW * w;      // S^T, then P^T | dS^T
        const uint32_t tB = tmem + lane_base + reg_s(gs + 1) + kCW * w;  // dP^T
        if (!wait_u(do_full + st, (gs / NSD) & 1) || !wait_u(q_full + sq, (gs / NSQ) & 1) ||
            !wait_u(s_full, gs & 1)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        // ---- P^T = exp2(S * scale*log2e - LSE*log2e) on this group's 32 query columns
        float pf[kCW];
        {
          uint32_t sv[kCW];
          tc::tmem_ld32(tA, sv);
          const float4* l4 = reinterpret_cast<const float4*>(sLSE + st * kB + kCW * w);
          tc::tmem_ld_wait();
          const int lo = j - (qb * kB + kCW * w);  // visible query columns: [lo, hi]
          const int hi = Ej - (qb * kB + kCW * w);
          const uint64_t sl2 = tc::f2(p.scale_log2, p.scale_log2), nl2 = tc::f2(-kLog2e, -kLog2e);
#pragma unroll
          for (int c4 = 0; c4 < kCW / 4; ++c4) {  // packed pairs: S*scale*log2e - LSE*log2e
            const float4 l = l4[c4];
            const int c = 4 * c4;
            const uint64_t a01 = tc::fma2(tc::f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2,
                                          tc::mul2(tc::f2(l.x, l.y), nl2));
            const uint64_t a23 = tc::fma2(tc::f2(__uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3])), sl2,
                                          tc::mul2(tc::f2(l.z, l.w), nl2));
            float x0, x1, x2, x3;
            tc::unf2(a01, x0, x1);
            tc::unf2(a23, x2, x3);
            pf[c] = tc::ex2(x0);
            pf[c + 1] = tc::ex2(x1);
            pf[c + 2] = tc::ex2(x2);
            pf[c + 3] = tc::ex2(x3);
          }
          if (!full) {
#pragma unroll
            for (int c = 0; c < kCW; ++c)
              if (c < lo || c > hi) pf[c] = 0.f;
          }
          uint32_t pw[kCW / 2];
#pragma unroll
          for (int e = 0; e < kCW / 2; ++e) pw[e] = tc::pack_bf16(pf[2 * e], pf[2 * e + 1]);
          tc::tmem_st16(tA, pw);  // first half of this group's S^T columns
          tc::tmem_st_wait();
        }
        tc::tc_fence_before();
        warp_arrive(p_ready);
        // ---- dS^T = P^T (dP^T - D)
        if (!wait_u(dp_full, gs & 1)) { ok = false; break; }
        tc::tc_fence_after();
        {
          uint32_t dpv[kCW];
          tc::tmem_ld32(tB, dpv);
          tc::tmem_ld_wait();
          tc::tc_fence_before();
          warp_arrive(dp_free);  // B_t may take S^T of the next step now
          const float4* d4 = reinterpret_cast<const float4*>(sDv + sq * kB + kCW * w);
          uint32_t dw[kCW / 2];
#pragma unroll
          for (int c4 = 0; c4 < kCW / 4; ++c4) {  // packed pairs: P (dP - D)
            const float4 dd = d4[c4];
            const int c = 4 * c4;
            const uint64_t g01 = tc::mul2(tc::f2(pf[c], pf[c + 1]),
                                          tc::sub2(tc::f2(__uint_as_float(dpv[c]), __uint_as_float(dpv[c + 1])),
                                                   tc::f2(dd.x, dd.y)));
            const uint64_t g23 = tc::mul2(tc::f2(pf[c + 2], pf[c + 3]),
                                          tc::sub2(tc::f2(__uint_as_float(dpv[c + 2]), __uint_as_float(dpv[c + 3])),
                                                   tc::f2(dd.z, dd.w)));
            float y0, y1, y2, y3;
            tc::unf2(g01, y0, y1);
            tc::unf2(g23, y2, y3);
            dw[2 * c4] = tc::pack_bf16(y0, y1);
            dw[2 * c4 + 1] = tc::pack_bf16(y2, y3);
          }
          tc::tmem_st16(tA + 16, dw);  // second half of this group's S^T columns
          tc::tmem_st_wait();
        }
        tc::tc_fence_before();
        warp_arrive(ds_ready);
      }
      if (!ok || !wait_u(acc_full, nk & 1)) { ok = false; break; }
      if (nk == 0) tc::grid_wait_prior();  // rows the preprocess zeroed are added into
      // ---- dK, dV rows of this key tile (warpgroup w: head-dim columns [w d/4, (w+1) d/4))
      tc::tc_fence_after();
      // A column longer than one item is split into several items that add
      // into zeroed fp32 rows: the outputs themselves for fp32 gradients, the
      // staging rows for bf16 gradients.
      const bool split = G * I.n_col > p.kv_chunk;
      const bool staged = !F32OUT && split;
      const int64_t off32 = (int64_t(krow + r) * p.hkv + I.g) * D + w * DW;  // fp32 row offset
#pragma unroll
      for (int c = 0; c < DW / 16; ++c) {
        uint32_t vv[16], kk[16];
        tc::tmem_ld16(tmem + lane_base + T_DV + w * DW + c * 16, vv);
        tc::tmem_ld16(tmem + lane_base + T_DK + w * DW + c * 16, kk);
        tc::tmem_ld_wait();
        if (staged) {
          store_row16<true>(reinterpret_cast<uint8_t*>(p.stage_v + off32 + c * 16), vv, 1.f, true);
          store_row16<true>(reinterpret_cast<uint8_t*>(p.stage_k + off32 + c * 16), kk, p.scale, true);
        } else {
          store_row16<F32OUT>(dv_row + c * 16 * ESZ, vv, 1.f, F32OUT && split, p.wide);
          store_row16<F32OUT>(dk_row + c * 16 * ESZ, kk, p.scale, F32OUT && split, p.wide);
        }
      }
      tc::tc_fence_before();
      warp_arrive(acc_free);
      if (staged) {
        // Every item maps this warp to the same 32-row x DW-column block of
        // the tile, so the warp that adds the column's last contribution to
        // its block converts that block's fp32 sums to bf16.  Its adds and
        // the other items' were made visible (fence) before each counted.
        __threadfence();
        __syncwarp();
        const uint32_t n_items = uint32_t((G * I.n_col + p.kv_chunk - 1) / p.kv_chunk);
        uint32_t done = 0;
        if ((threadIdx.x & 31) == 0)
          done = atomicAdd(p.kv_cnt + ((int64_t(I.b) * p.hkv + I.g) * p.n_blk + I.kb) * (4 * kNWG) + warp, 1u);
        done = __shfl_sync(0xffffffffu, done, 0);
        if (done == n_items - 1) {
          __threadfence();
#pragma unroll
          for (int c = 0; c < DW / 16; ++c) {
            uint32_t vv[16], kk[16];
            const float4* sv = reinterpret_cast<const float4*>(p.stage_v + off32 + c * 16);
            const float4* sk = reinterpret_cast<const float4*>(p.stage_k + off32 + c * 16);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float4 a = __ldcg(sv + e), b = __ldcg(sk + e);
              vv[4 * e] = __float_as_uint(a.x), vv[4 * e + 1] = __float_as_uint(a.y);
              vv[4 * e + 2] = __float_as_uint(a.z), vv[4 * e + 3] = __float_as_uint(a.w);
              kk[4 * e] = __float_as_uint(b.x), kk[4 * e + 1] = __float_as_uint(b.y);
              kk[4 * e + 2] = __float_as_uint(b.z), kk[4 * e + 3] = __float_as_uint(b.w);
            }
            store_row16<F32OUT>(dv_row + c * 16 * ESZ, vv, 1.f, false, p.wide);
            store_row16<F32OUT>(dk_row + c * 16 * ESZ, kk, 1.f, false, p.wide);  // scaled when added
          }
        }
      }
      qs += I.n;
      ++nk;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kWMma) tc::tmem_dealloc(tmem, 512);
  rearm_counter(p.sched + 2);
}

// =========================================================================== dQ kernel
//
// A step is one key tile j of the query tile's row.  TMEM: three 128-column
// regions R0..R2 and the dQ accumulator in [384, 384+D).  S(j) goes to
// R[j%3] and dP(j) to R[(j+1)%3]; compute warpgroup w owns key columns
// [32w, 32w+32) and writes dS(j) packed into the first 16 of its S columns.
// R[(j+1)%3] is free once dP(j) has been read, so S(j+1) and dP(j+1) (into
// R[(j+2)%3], whose dS(j-1) dQ(j-1) read before them) are issued then, ahead
// of dQ(j); the next tile's exponentials overlap dQ(j) and dP(j+1).

constexpr int kNIR = 4;  // dQ item ring slots: the producer publishes an item one ahead

template <int D>
struct DqCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = NCH * kChunk;  // 128-row tile of Q, dO, K or V
  static constexpr int NSK = D == 128 ? 3 : 6;    // K(j) is read by S(j) and again by dQ(j)
  static constexpr int NSV = D == 128 ? 2 : 4;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = TILE;
  static constexpr uint32_t OFF_K = 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + NSK * TILE;
  static constexpr uint32_t OFF_BAR = OFF_V + NSV * TILE;
  // q_full, q_empty, k_full[NSK], k_empty[NSK], v_full[NSV], v_empty[NSV], s_full, dp_full,
  // dp_free, ds_ready[2], dq_final, dq_free, drain, item_full[NIR], item_empty[NIR]
  static constexpr int NBAR = 2 + 2 * NSK + 2 * NSV + 8 + 2 * kNIR;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  // tmem slot, abort flag, then the item ring: kNIR x {index, n, e0, first CSR entry}
  static constexpr uint32_t OFF_RING = OFF_MISC + 16;
  static constexpr uint32_t BYTES = OFF_RING + kNIR * 16;  // base checked 1024-byte aligned
  static_assert(BYTES <= kSmemMax, "shared memory budget");
};

struct DqItem {
  int b, h, qb, e0, n;
  const int32_t* list;
};

__device__ __forceinline__ DqItem decode_dq(const BwdParams& p, int it) {
  DqItem r;
  const int per_b = p.hq * p.n_blk;
  r.b = it / per_b;
  const int rem = it - r.b * per_b;
  r.h = rem / p.n_blk;
  r.qb = p.n_blk - 1 - rem % p.n_blk;  // deepest (usually heaviest) query blocks first
  const int32_t* rp = p.q_ptr + r.b * (p.n_blk + 1);
  r.e0 = rp[r.qb];
  r.n = rp[r.qb + 1] - r.e0;
  r.list = p.q_idx + int64_t(r.b) * p.cap + r.e0;
  return r;
}

// (tree, query head, query block) of dQ item `it`, the index arithmetic of
// decode_dq without its CSR reads.
__device__ __forceinline__ void dq_coords(const BwdParams& p, int it, int& b, int& h, int& qb) {
  const int per_b = p.hq * p.n_blk;
  b = it / per_b;
  const int rem = it - b * per_b;
  h = rem / p.n_blk;
  qb = p.n_blk - 1 - rem % p.n_blk;
}

__device__ __forceinline__ uint32_t rot3(int j) { return uint32_t(j % 3) * 128u; }

template <int D, bool F32OUT>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const BwdParams p) {
  using C = DqCfg<D>;
  constexpr int NCH = C::NCH, NSK = C::NSK, NSV = C::NSV;
  constexpr uint32_t TILE = C::TILE;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (tc::smem_u32(smem) & 1023u) {  // uniform over the CTA: every thread leaves
    if (threadIdx.x == 0) atomicOr(&g_status_bwd, 2u);
    return;
  }
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bar;
  uint64_t* q_empty = bar + 1;
  uint64_t* k_full = bar + 2;
  uint64_t* k_empty = k_full + NSK;
  uint64_t* v_full = k_empty + NSK;
  uint64_t* v_empty = v_full + NSV;
  uint64_t* s_full = v_empty + NSV;
  uint64_t* dp_full = s_full + 1;
  uint64_t* dp_free = s_full + 2;
  uint64_t* ds_ready = s_full + 3;  // [2]: a fast thread may arrive for tile j+1 early
  uint64_t* dq_final = s_full + 5;
  uint64_t* dq_free = s_full + 6;
  uint64_t* drain = s_full + 7;
  uint64_t* item_full = s_full + 8;            // [kNIR]
  uint64_t* item_empty = s_full + 8 + kNIR;    // [kNIR]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* item_ring = reinterpret_cast<volatile int*>(smem + C::OFF_RING);  // [kNIR][4]

  const int warp = threadIdx.x >> 5;
  const int G = p.hq / p.hkv;
  constexpr uint32_t T_DQ = 384;
  constexpr int NCONS = 1 + 128 * kNWG;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    tc::mbar_init(q_empty, 1);
    for (int s = 0; s < NSK; ++s) {
      tc::mbar_init(k_full + s, 1);
      tc::mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < NSV; ++s) {
      tc::mbar_init(v_full + s, 1);
      tc::mbar_init(v_empty + s, 1);
    }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(dp_full, 1);
    tc::mbar_init(dp_free, 128 * kNWG);
    tc::mbar_init(ds_ready, 128 * kNWG);
    tc::mbar_init(ds_ready + 1, 128 * kNWG);
    tc::mbar_init(dq_final, 1);
    tc::mbar_init(dq_free, 128 * kNWG);
    tc::mbar_init(drain, 1);
    for (int s = 0; s < kNIR; ++s) {
      tc::mbar_init(item_full + s, 1);
      tc::mbar_init(item_empty + s, NCONS);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kWMma) tc::tmem_alloc(tmem_slot, 512);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto wait_u = [&](uint64_t* b_, uint32_t par) {
    return __all_sync(0xffffffffu, tc::mbar_wait(b_, par, abort_flag, &g_status_bwd));
  };

  if (warp == kWTma) {
    // ------------------------------------------------------------ producer
    // One thread runs the whole loop, like the MMA issuer: a warp-level sync
    // right after the bulk copies would hold the warp until they are issued.
    if (tc::elect_one()) {
    tc::tma_prefetch_desc(&tm_q);
    tc::tma_prefetch_desc(&tm_k);
    tc::tma_prefetch_desc(&tm_v);
    tc::tma_prefetch_desc(&tm_do);
    auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_bwd); };
    int gk = 0, gv = 0, nq = 0;  // K tiles, V tiles and Q tiles loaded so far
    bool ok = true;
    // Slot k of the ring gets the k-th item this CTA takes, decoded (index or
    // -1 once the items are used up, its tile count, CSR start and first
    // entry), so that no consumer reads the CSR at an item boundary.  Item
    // k + 1 is published while item k's tiles are still being loaded.
    auto take = [&](int k, DqItem& I) -> int {  // -2: aborted
      if (!wait1(item_empty + (k % kNIR), ((k / kNIR) & 1) ^ 1)) return -2;
      const uint32_t u = atomicAdd(p.sched + 4, 1u);
      const int it = u < uint32_t(p.dq_items) ? int(u) : -1;  // unsigned: no index below 0
      I.n = 0;
      if (it >= 0) I = decode_dq(p, it);
      const int first = I.n > 0 ? I.list[0] : 0;
      volatile int* slot = item_ring + 4 * (k % kNIR);
      slot[0] = it;
      slot[1] = I.n;
      slot[2] = it >= 0 ? I.e0 : 0;
      slot[3] = first;
      tc::mbar_arrive(item_full + (k % kNIR));
      return it;
    };
    DqItem I, J;
    int it = take(0, I);
    ok = it != -2;
    for (int k = 0; ok && it >= 0; ++k) {
      const int g = I.h / G;
      if (I.n > 0) {
        const int row0 = I.b * p.t_pad + I.qb * kB;
        if (!(ok = wait1(q_empty, (nq & 1) ^ 1))) break;
        tc::mbar_arrive_expect_tx(q_full, 2 * TILE);
        for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sQ + c * kChunk, &tm_q, q_full, c * 64, I.h, row0);
        for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sDO + c * kChunk, &tm_do, q_full, c * 64, I.h, row0);
        ++nq;
      }
      const int jt = take(k + 1, J);
      ok = jt != -2;
      if (!ok) break;
      if (jt >= 0 && J.n > 0) {  // the next item's Q and dO into L2 meanwhile
        const int nrow0 = J.b * p.t_pad + J.qb * kB;
        for (int c = 0; c < NCH; ++c) {
          tc::tma_prefetch_3d(&tm_q, c * 64, J.h, nrow0);
          tc::tma_prefetch_3d(&tm_do, c * 64, J.h, nrow0);
        }
      }
      int entry = I.n > 0 ? I.list[0] : 0;
      for (int j = 0; ok && j < I.n; ++j) {
        const int krow = I.b * p.t_pad + (entry >> 1) * kB;
        if (j + 1 < I.n) entry = I.list[j + 1];
        const int sk = gk % NSK;
        if (!(ok = wait1(k_empty + sk, ((gk / NSK) & 1) ^ 1))) break;
        tc::mbar_arrive_expect_tx(k_full + sk, TILE);
        for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sK + sk * TILE + c * kChunk, &tm_k, k_full + sk, c * 64, g, krow);
        ++gk;
        const int sv = gv % NSV;
        if (!(ok = wait1(v_empty + sv, ((gv / NSV) & 1) ^ 1))) break;
        tc::mbar_arrive_expect_tx(v_full + sv, TILE);
        for (int c = 0; c < NCH; ++c) tc::tma_load_3d(sV + sv * TILE + c * kChunk, &tm_v, v_full + sv, c * 64, g, krow);
        ++gv;
      }
      I = J;
      it = jt;
    }
    if (*abort_flag) {  // let the copies already issued land before the CTA exits
      volatile int never = 0;
      if (nq > 0) tc::mbar_wait(q_full, (nq - 1) & 1, &never, &g_status_bwd, 100000000ull);
      for (int jj = (gk > NSK ? gk - NSK : 0); jj < gk; ++jj)
        tc::mbar_wait(k_full + (jj % NSK), (jj / NSK) & 1, &never, &g_status_bwd, 100000000ull);
      for (int jj = (gv > NSV ? gv - NSV : 0); jj < gv; ++jj)
        tc::mbar_wait(v_full + (jj % NSV), (jj / NSV) & 1, &never, &g_status_bwd, 100000000ull);
    }
    }
    __syncwarp();
  } else if (warp == kWMma) {
    // ------------------------------------------------------------ MMA issuer
    // One thread runs the whole loop (a warp-level sync after tcgen05.mma
    // would hold the warp until the queued MMAs have gone into the pipe).
    constexpr uint32_t idesc_s = tc::idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_q = tc::idesc_bf16(128, D, false, true);
    const uint64_t dQ_ = tc::smem_desc(tc::smem_u32(sQ), 16, 1024);
    const uint64_t dDO_ = tc::smem_desc(tc::smem_u32(sDO), 16, 1024);
    const uint64_t dKk = tc::smem_desc(tc::smem_u32(sK), 16, 1024);      // K as K-major B
    const uint64_t dKm = tc::smem_desc(tc::smem_u32(sK), kChunk, 1024);  // K as MN-major B
    const uint64_t dV_ = tc::smem_desc(tc::smem_u32(sV), 16, 1024);
    auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_bwd); };
    auto issue_sdp = [&](int gt) -> bool {  // S(gt) = Q K^T into R[gt%3]; dP(gt) = dO V^T into R[(gt+1)%3]
      const int sk = gt % NSK, sv = gt % NSV;
      if (!wait1(k_full + sk, (gt / NSK) & 1)) return false;
      tc::tc_fence_after();
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        tc::mma_ss(tmem + rot3(gt), dQ_ + kslice(k), dKk + ((sk * TILE) >> 4) + kslice(k), idesc_s, k > 0);
      tc::mma_commit(s_full);
      if (!wait1(v_full + sv, (gt / NSV) & 1)) return false;
      tc::tc_fence_after();
#pragma unroll
      for (int k = 0; k < D / 16; ++k)
        tc::mma_ss(tmem + rot3(gt + 1), dDO_ + kslice(k), dV_ + ((sv * TILE) >> 4) + kslice(k), idesc_s, k > 0);
      tc::mma_commit(dp_full);
      tc::mma_commit(v_empty + sv);
      return true;
    };
    auto commit = [&](uint64_t* b_) { tc::mma_commit(b_); };
    if (tc::elect_one()) {
    int gt = 0, nq = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!(ok = wait1(item_full + (k % kNIR), (k / kNIR) & 1))) break;
      const int it = item_ring[4 * (k % kNIR)];
      const int n = item_ring[4 * (k % kNIR) + 1];
      tc::mbar_arrive(item_empty + (k % kNIR));
      if (it < 0) break;
      if (n == 0) continue;
      if (!(ok = wait1(q_full, nq & 1))) break;
      if (!(ok = issue_sdp(gt))) break;
      if (n == 1) commit(q_empty);  // Q and dO are read by S and dP only
      for (int j = 0; ok && j < n; ++j) {
        const int g = gt + j, sk = g % NSK;
        if (j + 1 < n) {  // the next tile's S and dP once dP(j) has been read
          if (!(ok = wait1(dp_free, g & 1))) break;
          if (!(ok = issue_sdp(g + 1))) break;
          if (j + 2 == n) commit(q_empty);
        }
        if (!(ok = wait1(ds_ready + (g & 1), (g >> 1) & 1))) break;
        if (j == 0 && nq > 0 && !(ok = wait1(dq_free, (nq - 1) & 1))) break;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kB / 16; ++kk)  // dQ += dS K, dS packed bf16 in R[g%3]
          mma_ts(tmem + T_DQ, packed_a(tmem + rot3(g), 0, kk), dKm + ((sk * TILE) >> 4) + ((kk * 2048) >> 4),
                 idesc_q, (j > 0 || kk > 0) ? 1u : 0u);
        tc::mma_commit(k_empty + sk);
      }
      if (!ok) break;
      commit(dq_final);
      gt += n;
      ++nq;
    }
    if (*abort_flag) {
      volatile int never = 0;
      tc::mma_commit(drain);
      tc::mbar_wait(drain, 0, &never, &g_status_bwd, 100000000ull);
    }
    }
    __syncwarp();
  } else if (warp < 4 * kNWG) {
    // ------------------------------------------------------------ compute warpgroups
    const int w = warp >> 2;          // key columns [32w, 32w+32) of each tile
    const int r = threadIdx.x & 127;  // query row = TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    constexpr int ESZ = F32OUT ? 4 : 2;
    constexpr int DW = D / kNWG;
    int gt = 0, nq = 0;
    bool ok = true;
    // The next item from the ring, with this thread's LSE, D and first mask
    // word requested before the current item's dQ stores go out (a load
    // issued behind 64 KB of stores waits for them to drain).
    struct Next {
      int it, n, e0, first;
      float lse, drow;
      uint32_t mk;
    };
    auto prefetch = [&](int k, Next& x) -> bool {
      if (!wait_u(item_full + (k % kNIR), (k / kNIR) & 1)) return false;
      const volatile int* slot = item_ring + 4 * (k % kNIR);
      x.it = slot[0];
      x.n = slot[1];
      x.e0 = slot[2];
      x.first = slot[3];
      tc::mbar_arrive(item_empty + (k % kNIR));
      x.lse = 0.f;
      x.drow = 0.f;
      x.mk = 0u;
      if (x.it >= 0 && x.n > 0) {
        int b, h, qb;
        dq_coords(p, x.it, b, h, qb);
        const int64_t vec = (int64_t(b) * p.hq + h) * p.t_pad + qb * kB + r;
        x.lse = p.lse[vec];
        x.drow = p.dvec[vec];
        if (!(x.first & 1))
          x.mk = reinterpret_cast<const uint32_t*>(p.qmask + (int64_t(b) * p.cap + x.e0) * kB + r)[w];
      }
      return true;
    };
    Next nx;
    ok = prefetch(0, nx);
    for (int k = 0; ok; ++k) {
      const Next I = nx;
      if (I.it < 0) break;
      int b, h, qb;
      dq_coords(p, I.it, b, h, qb);
      const int row0 = b * p.t_pad + qb * kB;
      uint8_t* dq_row = static_cast<uint8_t*>(p.dq) + ((int64_t(row0 + r) * p.hq + h) * D + w * DW) * ESZ;
      if (I.n == 0) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < DW * ESZ / 16; ++c) reinterpret_cast<uint4*>(dq_row)[c] = z;
        ok = prefetch(k + 1, nx);
        continue;
      }
      const float nlse = -I.lse * kLog2e;
      const uint64_t sl2 = tc::f2(p.scale_log2, p.scale_log2), nl2 = tc::f2(nlse, nlse);
      const uint64_t drow2 = tc::f2(I.drow, I.drow);
      const uint32_t* qmask_row =
          reinterpret_cast<const uint32_t*>(p.qmask + (int64_t(b) * p.cap + I.e0) * kB + r) + w;
      const int32_t* list = p.q_idx + int64_t(b) * p.cap + I.e0;
      int entry = I.first;
      uint32_t mk = I.mk;
      for (int j = 0; j < I.n; ++j) {
        const int g = gt + j;
        const bool full = entry & 1;
        const uint32_t mcur = mk;  // this group's 32 key columns
        if (j + 1 < I.n) {
          entry = list[j + 1];
          if (!(entry & 1)) mk = qmask_row[int64_t(j + 1) * kB * 4];
        }
        const uint32_t tS = tmem + lane_base + rot3(g) + kCW * w;
        if (!wait_u(s_full, g & 1)) { ok = false; break; }
        tc::tc_fence_after();
        float pf[kCW];
        {
          uint32_t sv[kCW];
          tc::tmem_ld32(tS, sv);
          tc::tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < kCW; c += 2) {  // packed pairs: S*scale*log2e - LSE*log2e
            float x0, x1;
            tc::unf2(tc::fma2(tc::f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2, nl2), x0, x1);
            pf[c] = tc::ex2(x0);
            pf[c + 1] = tc::ex2(x1);
          }
          if (!full) {
#pragma unroll
            for (int c = 0; c < kCW; ++c)
              if (!((mcur >> c) & 1u)) pf[c] = 0.f;
          }
        }
        if (!wait_u(dp_full, g & 1)) { ok = false; break; }
        tc::tc_fence_after();
        {
          uint32_t dpv[kCW];
          tc::tmem_ld32(tmem + lane_base + rot3(g + 1) + kCW * w, dpv);
          tc::tmem_ld_wait();
          tc::tc_fence_before();
          tc::mbar_arrive(dp_free);  // R[(g+1)%3] may take S of the next tile now
          uint32_t dw[kCW / 2];
#pragma unroll
          for (int e = 0; e < kCW / 2; ++e) {  // packed pairs: P (dP - D)
            float y0, y1;
            tc::unf2(tc::mul2(tc::f2(pf[2 * e], pf[2 * e + 1]),
                              tc::sub2(tc::f2(__uint_as_float(dpv[2 * e]), __uint_as_float(dpv[2 * e + 1])), drow2)),
                     y0, y1);
            dw[e] = tc::pack_bf16(y0, y1);
          }
          tc::tmem_st16(tS, dw);  // dS over the first half of this group's S columns
          tc::tmem_st_wait();
        }
        tc::tc_fence_before();
        tc::mbar_arrive(ds_ready + (g & 1));
      }
      if (!ok || !prefetch(k + 1, nx) || !wait_u(dq_final, nq & 1)) { ok = false; break; }
      tc::tc_fence_after();
      if constexpr (DW == 32) {  // one TMEM load for the thread's 32 columns
        uint32_t v[32];
        tc::tmem_ld32(tmem + lane_base + T_DQ + w * DW, v);
        tc::tmem_ld_wait();
        tc::tc_fence_before();
        tc::mbar_arrive(dq_free);  // the stores below read registers only
#pragma unroll
        for (int c = 0; c < 2; ++c)
          store_row16<F32OUT>(dq_row + c * 16 * ESZ, reinterpret_cast<const uint32_t(&)[16]>(v[16 * c]), p.scale,
                              false, p.wide);
      } else {
#pragma unroll
        for (int c = 0; c < DW / 16; ++c) {
          uint32_t v[16];
          tc::tmem_ld16(tmem + lane_base + T_DQ + w * DW + c * 16, v);
          tc::tmem_ld_wait();
          store_row16<F32OUT>(dq_row + c * 16 * ESZ, v, p.scale, false, p.wide);
        }
        tc::tc_fence_before();
        tc::mbar_arrive(dq_free);
      }
      gt += I.n;
      ++nq;
    }
  }

  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == kWMma) tc::tmem_dealloc(tmem, 512);
  rearm_counter(p.sched + 4);
}

// =========================================================================== dQ kernel, head pairs
//
// For d = 128 and GQA groups of an even number of query heads, a cluster of
// two CTAs (the two SMs of a TPC) takes one (query tile, head pair, tree)
// item, CTA c computing query head 2p + c.  Both heads read the same key and
// value head, so every MMA of the step runs once over the pair with M = 256
// (cta_group::2): each CTA keeps its own Q and dO tiles and its own rows of
// S, dP, dS and dQ in TMEM exactly as above, but only half of each B
// operand -- keys [64c, 64c+64) of the K and V tiles for S and dP, and
// head-dim columns [64c, 64c+64) of the K tile for dQ.  Per 128x128x16 MMA a
// CTA reads 6 KB of shared memory instead of 8 KB, and per step it loads
// 48 KB of K and V instead of 64 KB: the MMAs are no longer held back by
// shared-memory bandwidth.  The even CTA fetches the items and issues every
// MMA; the copies of both CTAs complete on its barriers, its MMA completions
// are multicast to both CTAs, and each compute warp signals it once.
//
// TMEM (per CTA): S in [0, 128), dP in [128, 256), packed dS in [256, 320),
// the item's dO tile in [320, 384) and the dQ accumulator in [384, 512).
// S(j+1) is issued as soon as the compute warps have read S(j), at the
// start of step j's exponentials, dP(j+1) once they have read dP(j), and
// dQ(j) once dS(j) is packed; an MMA's completion is only seen a few hundred
// cycles after its issue, and this order keeps the next step's S and dP
// ahead of the compute warps, so that the tensor pipe, not that latency,
// sets the pace.  S and dP are issued by one warp, dQ by another.  At an
// item's start its dO tile is copied from shared memory into TMEM (the A
// operand of its dP MMAs), which frees the single shared-memory dO buffer at
// once: the next item's dO is loaded a whole item ahead, and an item's first
// dP does not wait for it.

constexpr int kNWarpsC = 4 * kNWG;  // compute warps per CTA
// One MMA takes 64 cycles of the pair's tensor pipes but about as long to
// issue from one thread, so two warps issue: one S and dP, one dQ (they
// touch disjoint TMEM and are ordered through the compute warps' signals).
constexpr int kWMmaQ = kWMma + 1;
constexpr int kThreads2 = kThreads + 32;

template <int D>
struct Dq2Cfg {
  static_assert(D == 128, "head pairs: d = 128");
  static constexpr uint32_t TILE = 2 * kChunk;   // Q or dO tile, 128 rows x 128 columns
  static constexpr uint32_t PIECE = kChunk / 2;  // 64 rows x 64 columns
  // K stage: [my 64 keys x columns 0-63 | my keys x 64-127 | keys 0-63 x my column half |
  // keys 64-127 x my column half]; V stage: my keys x both column halves.
  static constexpr uint32_t KST = 4 * PIECE;
  static constexpr uint32_t VST = 2 * PIECE;
  // Two Q buffers: the next item's Q lands while this item runs, so its
  // first S is issued as soon as this item's last S has been read.
  static constexpr int NSQ = 2, NSK = 3, NSV = 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_DO = NSQ * TILE;
  static constexpr uint32_t OFF_K = OFF_DO + TILE;
  static constexpr uint32_t OFF_V = OFF_K + NSK * KST;
  static constexpr uint32_t OFF_BAR = OFF_V + NSV * VST;
  // q_full[NSQ], q_empty[NSQ], do_full, do_empty, k_full[NSK], k_empty[NSK], v_full[NSV],
  // v_empty[NSV], s_full, dp_full, s_free, dp_free, ds_ready[2], ds_free[2], dq_final, dq_free,
  // drain[2], item_full[NIR], item_empty[NIR]
  static constexpr int NBAR = 2 * NSQ + 2 + 2 * NSK + 2 * NSV + 12 + 2 * kNIR;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t OFF_RING = OFF_MISC + 16;  // kNIR x {index, n, e0, first CSR entry}
  static constexpr uint32_t BYTES = OFF_RING + kNIR * 16;
  static_assert(BYTES <= kSmemMax, "shared memory budget");
};

// (tree, head pair, query block) of pair item `it`, in decode_dq's order.
__device__ __forceinline__ void dq2_coords(const BwdParams& p, int it, int& b, int& hp, int& qb) {
  const int per_b = (p.hq >> 1) * p.n_blk;
  b = it / per_b;
  const int rem = it - b * per_b;
  hp = rem / p.n_blk;
  qb = p.n_blk - 1 - rem % p.n_blk;
}

template <int D, bool F32OUT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads2, 1)
    attn_bwd_dq2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k64,
                        const __grid_constant__ CUtensorMap tm_v64, const __grid_constant__ CUtensorMap tm_do,
                        const BwdParams p) {
  using C = Dq2Cfg<D>;
  constexpr int NSQ = C::NSQ, NSK = C::NSK, NSV = C::NSV;
  constexpr uint32_t TILE = C::TILE, PIECE = C::PIECE, KST = C::KST, VST = C::VST;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if (tc::smem_u32(smem) & 1023u) {  // the same for every CTA of the launch: all leave
    if (threadIdx.x == 0) atomicOr(&g_status_bwd, 2u);
    return;
  }
  const uint32_t crank = tc::cta_rank();
  const bool lead = crank == 0;
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sDO = smem + C::OFF_DO;
  uint8_t* sK = smem + C::OFF_K;
  uint8_t* sV = smem + C::OFF_V;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bar;              // [NSQ]
  uint64_t* q_empty = bar + NSQ;       // [NSQ]
  uint64_t* do_full = bar + 2 * NSQ;
  uint64_t* do_empty = do_full + 1;
  uint64_t* k_full = do_full + 2;
  uint64_t* k_empty = k_full + NSK;
  uint64_t* v_full = k_empty + NSK;
  uint64_t* v_empty = v_full + NSV;
  uint64_t* s_full = v_empty + NSV;
  uint64_t* dp_full = s_full + 1;
  uint64_t* s_free = s_full + 2;
  uint64_t* dp_free = s_full + 3;
  uint64_t* ds_ready = s_full + 4;  // (one packed-dS buffer: slot 5 is unused)
  uint64_t* ds_free = s_full + 6;   // (slot 7 is unused)
  uint64_t* dq_final = s_full + 8;
  uint64_t* dq_free = s_full + 9;
  uint64_t* drain = s_full + 10;              // [2]: one per issuing warp
  uint64_t* item_full = s_full + 12;          // [kNIR]
  uint64_t* item_empty = s_full + 12 + kNIR;  // [kNIR]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* item_ring = reinterpret_cast<volatile int*>(smem + C::OFF_RING);  // [kNIR][4]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.hq / p.hkv;
  constexpr uint32_t T_S = 0, T_DP = 128, T_DS = 256, T_DO = 320, T_DQ = 384;
  // item-slot consumers, all arriving on the even CTA: its two MMA warps and
  // compute warps, the odd CTA's producer and compute warps
  constexpr int NCONS2 = 2 * (1 + kNWarpsC) + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NSQ; ++s) {
      tc::mbar_init(q_full + s, 1);
      tc::mbar_init(q_empty + s, 1);
    }
    tc::mbar_init(do_full, 1);
    tc::mbar_init(do_empty, 1);
    for (int s = 0; s < NSK; ++s) {
      tc::mbar_init(k_full + s, 1);
      tc::mbar_init(k_empty + s, 1);
    }
    for (int s = 0; s < NSV; ++s) {
      tc::mbar_init(v_full + s, 1);
      tc::mbar_init(v_empty + s, 1);
    }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(dp_full, 1);
    tc::mbar_init(s_free, 2 * kNWarpsC);
    tc::mbar_init(dp_free, 2 * kNWarpsC);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(ds_ready + s, 2 * kNWarpsC);
      tc::mbar_init(ds_free + s, 1);
    }
    tc::mbar_init(dq_final, 1);
    tc::mbar_init(dq_free, 2 * kNWarpsC);
    tc::mbar_init(drain, 1);
    tc::mbar_init(drain + 1, 1);
    for (int s = 0; s < kNIR; ++s) {
      tc::mbar_init(item_full + s, 1);
      tc::mbar_init(item_empty + s, NCONS2);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kWMma) tc::tmem_alloc2(tmem_slot, 512);
  tc::tc_fence_before();
  tc::cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto wait_u = [&](uint64_t* b_, uint32_t par) {
    return __all_sync(0xffffffffu, tc::mbar_wait(b_, par, abort_flag, &g_status_bwd));
  };
  auto wait_ring = [&](uint64_t* b_, uint32_t par) {  // item slots: written across the pair
    return __all_sync(0xffffffffu, tc::mbar_wait_cluster(b_, par, abort_flag, &g_status_bwd));
  };
  // one arrival per warp on the even CTA's copy of `b_` (after the warp's own tcgen05 fences)
  auto warp_arrive_lead = [&](uint64_t* b_) {
    __syncwarp();
    if (lane == 0) tc::mbar_arrive_remote(tc::peer_addr(b_, 0));
    __syncwarp();
  };

  if (warp == kWTma) {
    // ------------------------------------------------------------ producers (both CTAs)
    // One thread runs the whole loop, like the MMA issuers: a warp-level sync
    // right after the bulk copies would hold the warp until they are issued.
    if (tc::elect_one()) {
    tc::tma_prefetch_desc(&tm_q);
    tc::tma_prefetch_desc(&tm_k64);
    tc::tma_prefetch_desc(&tm_v64);
    tc::tma_prefetch_desc(&tm_do);
    auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_bwd); };
    int gk = 0, gv = 0, nq = 0;
    bool ok = true;
    struct Item {
      int it, n, e0;
    };
    // Even CTA: slot k gets the k-th item the pair takes, written into both
    // CTAs' rings, one item ahead of the loads.  Odd CTA: reads slot k.
    auto take = [&](int k, Item& I) -> bool {
      const int slot = k % kNIR;
      if (!wait1(item_empty + slot, ((k / kNIR) & 1) ^ 1)) return false;
      const uint32_t u = atomicAdd(p.sched + 4, 1u);
      I.it = u < uint32_t(p.dq_items) ? int(u) : -1;  // unsigned: no index below 0
      I.n = 0;
      I.e0 = 0;
      int first = 0;
      if (I.it >= 0) {
        int b, hp, qb;
        dq2_coords(p, I.it, b, hp, qb);
        const int32_t* rp = p.q_ptr + b * (p.n_blk + 1);
        I.e0 = rp[qb];
        I.n = rp[qb + 1] - I.e0;
        if (I.n > 0) first = p.q_idx[int64_t(b) * p.cap + I.e0];
      }
      volatile int* mine = item_ring + 4 * slot;
      mine[0] = I.it;
      mine[1] = I.n;
      mine[2] = I.e0;
      mine[3] = first;
      const uint32_t peer = tc::peer_addr(const_cast<int*>(mine), 1);
      tc::st_cluster_u32(peer, uint32_t(I.it));
      tc::st_cluster_u32(peer + 4, uint32_t(I.n));
      tc::st_cluster_u32(peer + 8, uint32_t(I.e0));
      tc::st_cluster_u32(peer + 12, uint32_t(first));
      tc::mbar_arrive(item_full + slot);
      tc::mbar_arrive_release_cluster(tc::peer_addr(item_full + slot, 1));  // after the ring stores
      return true;
    };
    auto read = [&](int k, Item& I) -> bool {
      const int slot = k % kNIR;
      if (!tc::mbar_wait_cluster(item_full + slot, (k / kNIR) & 1, abort_flag, &g_status_bwd)) return false;
      I.it = item_ring[4 * slot];
      I.n = item_ring[4 * slot + 1];
      I.e0 = item_ring[4 * slot + 2];
      tc::mbar_arrive_remote(tc::peer_addr(item_empty + slot, 0));  // this warp's one arrival
      return true;
    };
    // Q of an item goes into buffer (count of loaded Q tiles) % NSQ; it is
    // requested as soon as the item is known, one item ahead of its K/V.
    int nd = 0;  // dO tiles loaded
    auto load_q = [&](const Item& X) -> bool {
      int xb, xhp, xqb;
      dq2_coords(p, X.it, xb, xhp, xqb);
      const int qs = nq % NSQ;
      if (!wait1(q_empty + qs, ((nq / NSQ) & 1) ^ 1)) return false;
      if (lead) tc::mbar_arrive_expect_tx(q_full + qs, 2 * TILE);  // Q of both CTAs
      const uint32_t lb = tc::peer_addr(q_full + qs, 0);
      for (int c = 0; c < 2; ++c)
        tc::tma_load_3d_pair(sQ + qs * TILE + c * kChunk, &tm_q, lb, c * 64, 2 * xhp + int(crank),
                             xb * p.t_pad + xqb * kB);
      ++nq;
      return true;
    };
    // dO of an item goes into the one shared-memory buffer, which frees as
    // soon as the item's start has copied it into TMEM.
    auto load_do = [&](const Item& X) -> bool {
      int xb, xhp, xqb;
      dq2_coords(p, X.it, xb, xhp, xqb);
      if (!wait1(do_empty, (nd & 1) ^ 1)) return false;
      if (lead) tc::mbar_arrive_expect_tx(do_full, 2 * TILE);  // dO of both CTAs
      const uint32_t lb = tc::peer_addr(do_full, 0);
      for (int c = 0; c < 2; ++c)
        tc::tma_load_3d_pair(sDO + c * kChunk, &tm_do, lb, c * 64, 2 * xhp + int(crank), xb * p.t_pad + xqb * kB);
      ++nd;
      return true;
    };
    Item I, J;
    ok = lead ? take(0, I) : read(0, I);
    if (ok && I.it >= 0 && I.n > 0) ok = load_q(I) && load_do(I);
    for (int k = 0; ok && I.it >= 0; ++k) {
      int b, hp, qb;
      dq2_coords(p, I.it, b, hp, qb);
      const int g = (2 * hp) / G;
      // The next item's Q and dO after this item's first K and V tiles, so
      // that this item's first S and dP do not wait behind them.
      auto load_next = [&]() -> bool {
        if (!(lead ? take(k + 1, J) : read(k + 1, J))) return false;
        if (J.it >= 0 && J.n > 0 && !(load_q(J) && load_do(J))) return false;
        return true;
      };
      if (I.n == 0 && !(ok = load_next())) break;
      const int32_t* list = p.q_idx + int64_t(b) * p.cap + I.e0;
      int entry = I.n > 0 ? list[0] : 0;
      for (int j = 0; ok && j < I.n; ++j) {
        const int krow = b * p.t_pad + (entry >> 1) * kB;
        if (j + 1 < I.n) entry = list[j + 1];
        const int sk = gk % NSK;
        if (!(ok = wait1(k_empty + sk, ((gk / NSK) & 1) ^ 1))) break;
        {
          if (lead) tc::mbar_arrive_expect_tx(k_full + sk, 2 * KST);
          const uint32_t lb = tc::peer_addr(k_full + sk, 0);
          uint8_t* st = sK + sk * KST;
          const int mine = krow + 64 * int(crank);
          tc::tma_load_3d_pair(st, &tm_k64, lb, 0, g, mine);                       // my keys, columns 0-63
          tc::tma_load_3d_pair(st + PIECE, &tm_k64, lb, 64, g, mine);              // my keys, columns 64-127
          tc::tma_load_3d_pair(st + 2 * PIECE, &tm_k64, lb, 64 * int(crank), g, krow);       // keys 0-63
          tc::tma_load_3d_pair(st + 3 * PIECE, &tm_k64, lb, 64 * int(crank), g, krow + 64);  // keys 64-127
        }
        ++gk;
        const int sv = gv % NSV;
        if (!(ok = wait1(v_empty + sv, ((gv / NSV) & 1) ^ 1))) break;
        {
          if (lead) tc::mbar_arrive_expect_tx(v_full + sv, 2 * VST);
          const uint32_t lb = tc::peer_addr(v_full + sv, 0);
          uint8_t* st = sV + sv * VST;
          const int mine = krow + 64 * int(crank);
          tc::tma_load_3d_pair(st, &tm_v64, lb, 0, g, mine);
          tc::tma_load_3d_pair(st + PIECE, &tm_v64, lb, 64, g, mine);
        }
        ++gv;
        if (j == 0 && !(ok = load_next())) break;
      }
      if (!ok) break;
      I = J;
    }
    if (*abort_flag) {  // copies into this CTA's shared memory complete on the even CTA's barriers:
      const long long t0 = clock64();  // give any still in flight time to land before the CTA leaves
      while (clock64() - t0 < 400000) {
      }
    }
    }
    __syncwarp();
  } else if (warp == kWMma) {
    // ------------------------------------------------------------ S and dP issuer (even CTA)
    // Each issuer is one thread running the whole loop: a warp-level sync
    // after tcgen05.mma holds the warp until the thread's queued MMAs have
    // gone into the pipe, which would leave the pipe idle during its waits.
    if (lead && tc::elect_one()) {
      constexpr uint32_t idesc_s = tc::idesc_bf16(256, 128, false, false);
      const uint64_t dQ_ = tc::smem_desc(tc::smem_u32(sQ), 16, 1024);
      const uint64_t dDO_ = tc::smem_desc(tc::smem_u32(sDO), 16, 1024);
      const uint64_t dKx = tc::smem_desc(tc::smem_u32(sK), 16, 1024);               // my keys, K-major B
      const uint64_t dVx = tc::smem_desc(tc::smem_u32(sV), 16, 1024);
      auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_bwd); };
      auto issue_s = [&](int gt, int qs) -> bool {  // S(gt) = Q K^T over the pair, Q in buffer qs
        const int sk = gt % NSK;
        if (!wait1(k_full + sk, (gt / NSK) & 1)) return false;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc::mma2_ss(tmem + T_S, dQ_ + ((qs * TILE) >> 4) + kslice(k), dKx + ((sk * KST) >> 4) + kslice(k, PIECE),
                      idesc_s, k > 0);
        tc::mma2_commit_both(s_full);
        return true;
      };
      auto issue_dp = [&](int gt) -> bool {  // dP(gt) = dO V^T over the pair, dO in TMEM
        const int sv = gt % NSV;
        if (!wait1(v_full + sv, (gt / NSV) & 1)) return false;
        tc::tc_fence_after();
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
          tc::mma2_ts(tmem + T_DP, tmem + T_DO + 8 * k, dVx + ((sv * VST) >> 4) + kslice(k, PIECE), idesc_s, k > 0);
        tc::mma2_commit_both(dp_full);
        tc::mma2_commit_both(v_empty + sv);
        return true;
      };
      int gt = 0, nq = 0;
      auto commit = [&](uint64_t* b_) { tc::mma2_commit_both(b_); };
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (!(ok = tc::mbar_wait_cluster(item_full + (k % kNIR), (k / kNIR) & 1, abort_flag, &g_status_bwd))) break;
        const int it = item_ring[4 * (k % kNIR)];
        const int n = item_ring[4 * (k % kNIR) + 1];
        tc::mbar_arrive(item_empty + (k % kNIR));
        if (it < 0) break;
        if (n == 0) continue;
        // the previous item's last S and dP have been read (waited below)
        const int qs = nq % NSQ;
        if (!(ok = wait1(q_full + qs, (nq / NSQ) & 1))) break;
        if (!(ok = issue_s(gt, qs))) break;
        if (n == 1) commit(q_empty + qs);  // Q is read by S only
        // dO(k) into TMEM: the previous item's last dP has been read (dp_free
        // below), so the region its A operand came from is free
        if (!(ok = wait1(do_full, nq & 1))) break;
        tc::tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) tc::tmem_cp2_128x256b(tmem + T_DO + 8 * kk, dDO_ + kslice(kk));
        commit(do_empty);  // the buffer takes the next item's dO once the copy is done
        if (!(ok = issue_dp(gt))) break;
        for (int j = 0; ok && j < n; ++j) {
          const int g = gt + j;
          if (!(ok = wait1(s_free, g & 1))) break;
          if (j + 1 < n) {
            if (!(ok = issue_s(g + 1, qs))) break;
            if (j + 2 == n) commit(q_empty + qs);
          }
          if (!(ok = wait1(dp_free, g & 1))) break;
          if (j + 1 < n && !(ok = issue_dp(g + 1))) break;
        }
        if (!ok) break;
        gt += n;
        ++nq;
      }
      if (*abort_flag) {
        volatile int never = 0;
        tc::mma2_commit_both(drain);
        tc::mbar_wait(drain, 0, &never, &g_status_bwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == kWMmaQ) {
    // ------------------------------------------------------------ dQ issuer (even CTA)
    if (lead && tc::elect_one()) {
      auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_bwd); };
      constexpr uint32_t idesc_q = tc::idesc_bf16(256, D, false, true);
      const uint64_t dKy = tc::smem_desc(tc::smem_u32(sK + 2 * PIECE), kChunk, 1024);  // my columns, MN-major B
      int gt = 0, nq = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (!(ok = tc::mbar_wait_cluster(item_full + (k % kNIR), (k / kNIR) & 1, abort_flag, &g_status_bwd))) break;
        const int it = item_ring[4 * (k % kNIR)];
        const int n = item_ring[4 * (k % kNIR) + 1];
        tc::mbar_arrive(item_empty + (k % kNIR));
        if (it < 0) break;
        if (n == 0) continue;
        for (int j = 0; ok && j < n; ++j) {
          const int g = gt + j, sk = g % NSK;
          if (!(ok = wait1(ds_ready, g & 1))) break;
          if (j == 0 && nq > 0 && !(ok = wait1(dq_free, (nq - 1) & 1))) break;
          tc::tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kB / 16; ++kk)  // dQ += dS K over the pair, dS packed in T_DS
            tc::mma2_ts(tmem + T_DQ, tmem + T_DS + 8 * kk, dKy + ((sk * KST) >> 4) + ((kk * 2048) >> 4), idesc_q,
                        (j > 0 || kk > 0) ? 1u : 0u);
          tc::mma2_commit_both(ds_free);
          tc::mma2_commit_both(k_empty + sk);  // S(g) was read before dS(g) existed
        }
        if (!ok) break;
        tc::mma2_commit_both(dq_final);
        gt += n;
        ++nq;
      }
      if (*abort_flag) {
        volatile int never = 0;
        tc::mma2_commit_both(drain + 1);
        tc::mbar_wait(drain + 1, 0, &never, &g_status_bwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp < kNWarpsC) {
    // ------------------------------------------------------------ compute warpgroups (both CTAs)
    const int w = warp >> 2;          // key columns [32w, 32w+32) of each tile
    const int r = threadIdx.x & 127;  // query row = TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    constexpr int ESZ = F32OUT ? 4 : 2;
    constexpr int DW = D / kNWG;
    int gt = 0, nq = 0;
    bool ok = true;
    struct Next {
      int it, n, e0, first;
      float lse, drow;
      uint32_t mk;
    };
    auto prefetch = [&](int k, Next& x) -> bool {
      const int slot = k % kNIR;
      if (!wait_ring(item_full + slot, (k / kNIR) & 1)) return false;
      x.it = item_ring[4 * slot];
      x.n = item_ring[4 * slot + 1];
      x.e0 = item_ring[4 * slot + 2];
      x.first = item_ring[4 * slot + 3];
      warp_arrive_lead(item_empty + slot);
      x.lse = 0.f;
      x.drow = 0.f;
      x.mk = 0u;
      if (x.it >= 0 && x.n > 0) {
        int b, hp, qb;
        dq2_coords(p, x.it, b, hp, qb);
        const int64_t vec = (int64_t(b) * p.hq + 2 * hp + int(crank)) * p.t_pad + qb * kB + r;
        x.lse = p.lse[vec];
        x.drow = p.dvec[vec];
        if (!(x.first & 1))
          x.mk = reinterpret_cast<const uint32_t*>(p.qmask + (int64_t(b) * p.cap + x.e0) * kB + r)[w];
      }
      return true;
    };
    // An item's dQ is read out during the next item's first tile, after its
    // exponentials: the 64 KB of stores then drain while that tile's dP is
    // still loading instead of holding up its S (loads and barrier waits
    // issued behind a burst of stores wait for it).
    uint8_t* pend_row = nullptr;
    int pend_nq = 0;
    auto readout = [&]() -> bool {
      if (!wait_u(dq_final, pend_nq & 1)) return false;
      tc::tc_fence_after();
      uint32_t v[32];
      tc::tmem_ld32(tmem + lane_base + T_DQ + w * DW, v);
      tc::tmem_ld_wait();
      tc::tc_fence_before();
      warp_arrive_lead(dq_free);
#pragma unroll
      for (int c = 0; c < 2; ++c)
        store_row16<F32OUT>(pend_row + c * 16 * ESZ, reinterpret_cast<const uint32_t(&)[16]>(v[16 * c]), p.scale,
                            false, p.wide);
      pend_row = nullptr;
      return true;
    };
    Next nx;
    ok = prefetch(0, nx);
    for (int k = 0; ok; ++k) {
      const Next I = nx;
      if (I.it < 0) break;
      int b, hp, qb;
      dq2_coords(p, I.it, b, hp, qb);
      const int h = 2 * hp + int(crank);
      const int row0 = b * p.t_pad + qb * kB;
      uint8_t* dq_row = static_cast<uint8_t*>(p.dq) + ((int64_t(row0 + r) * p.hq + h) * D + w * DW) * ESZ;
      if (I.n == 0) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < DW * ESZ / 16; ++c) reinterpret_cast<uint4*>(dq_row)[c] = z;
        ok = prefetch(k + 1, nx);
        continue;
      }
      const float nlse = -I.lse * kLog2e;
      const uint64_t sl2 = tc::f2(p.scale_log2, p.scale_log2), nl2 = tc::f2(nlse, nlse);
      const uint64_t drow2 = tc::f2(I.drow, I.drow);
      const uint32_t* qmask_row =
          reinterpret_cast<const uint32_t*>(p.qmask + (int64_t(b) * p.cap + I.e0) * kB + r) + w;
      const int32_t* list = p.q_idx + int64_t(b) * p.cap + I.e0;
      int entry = I.first;
      uint32_t mk = I.mk;
      for (int j = 0; j < I.n; ++j) {
        const int g = gt + j;
        const bool full = entry & 1;
        const uint32_t mcur = mk;
        if (j + 1 < I.n) {
          entry = list[j + 1];
          if (!(entry & 1)) mk = qmask_row[int64_t(j + 1) * kB * 4];
        }
        if (!wait_u(s_full, g & 1)) { ok = false; break; }
        tc::tc_fence_after();
        float pf[kCW];
        {
          uint32_t sv[kCW];
          tc::tmem_ld32(tmem + lane_base + T_S + kCW * w, sv);
          tc::tmem_ld_wait();
          tc::tc_fence_before();
          warp_arrive_lead(s_free);  // S of the next tile may be issued now
#pragma unroll
          for (int c = 0; c < kCW; c += 2) {  // packed pairs: S*scale*log2e - LSE*log2e
            float x0, x1;
            tc::unf2(tc::fma2(tc::f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2, nl2), x0, x1);
            pf[c] = tc::ex2(x0);
            pf[c + 1] = tc::ex2(x1);
          }
          if (!full) {
#pragma unroll
            for (int c = 0; c < kCW; ++c)
              if (!((mcur >> c) & 1u)) pf[c] = 0.f;
          }
        }
        if (j == 0 && pend_row != nullptr && !readout()) { ok = false; break; }
        if (!wait_u(dp_full, g & 1)) { ok = false; break; }
        tc::tc_fence_after();
        {
          uint32_t dpv[kCW];
          tc::tmem_ld32(tmem + lane_base + T_DP + kCW * w, dpv);
          tc::tmem_ld_wait();
          tc::tc_fence_before();
          warp_arrive_lead(dp_free);
          uint32_t dw[kCW / 2];
#pragma unroll
          for (int e = 0; e < kCW / 2; ++e) {  // packed pairs: P (dP - D)
            float y0, y1;
            tc::unf2(tc::mul2(tc::f2(pf[2 * e], pf[2 * e + 1]),
                              tc::sub2(tc::f2(__uint_as_float(dpv[2 * e]), __uint_as_float(dpv[2 * e + 1])), drow2)),
                     y0, y1);
            dw[e] = tc::pack_bf16(y0, y1);
          }
          // dS(g) goes where dS(g-1) was: wait until dQ(g-1) has read it
          if (g >= 1 && !wait_u(ds_free, (g - 1) & 1)) { ok = false; break; }
          tc::tc_fence_after();
          tc::tmem_st16(tmem + lane_base + T_DS + 16 * w, dw);
          tc::tmem_st_wait();
        }
        tc::tc_fence_before();
        warp_arrive_lead(ds_ready);
      }
      if (!ok || !prefetch(k + 1, nx)) { ok = false; break; }
      pend_row = dq_row;
      pend_nq = nq;
      gt += I.n;
      ++nq;
    }
    if (ok && pend_row != nullptr) readout();  // the CTA's last item
  }

  tc::tc_fence_before();
  tc::cluster_sync();  // the pair's MMAs into either CTA's TMEM are done before it is freed
  tc::tc_fence_after();
  if (warp == kWMma) tc::tmem_dealloc2(tmem, 512);
  rearm_counter(p.sched + 4);
  // launched behind the KV kernel with programmatic serialization: do not
  // complete before it, so that work after this launch sees both finished
  tc::grid_wait_prior();
}

// D[b, h, i] = sum_d dO * O (fp32) for real rows, 0 for pad rows.  The
// [B*T*Hq, D] bf16 rows of O and dO are read with 16-byte loads, four per
// lane in flight: a warp covers 128 * 32 / D rows per pass, D / 8 lanes per
// row, and sums each row with shuffles.  It also zeroes the fp32 rows that
// the KV kernel's split columns add into: with fp32 gradients the dK and dV
// rows themselves (and those of the key tiles no query sees, which no item
// visits), with bf16 gradients the staging rows and the per-warp item
// counters; every other row is written whole by its single item.
// Four CTAs an SM: 64 registers a thread instead of 80 (three CTAs), which
// keeps a third more loads in flight (152 -> 142 us on the GRPO-shaped batch).
template <int D>
__global__ void __launch_bounds__(256, 4) bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                     const __nv_bfloat16* __restrict__ dout,
                                                     const int32_t* __restrict__ n_tokens, int32_t t_pad,
                                                     int32_t hq, int64_t n_rows, float* __restrict__ dvec,
                                                     float4* __restrict__ dk, float4* __restrict__ dv,
                                                     const int32_t* __restrict__ k_ptr, int32_t n_trees,
                                                     int32_t n_blk, int32_t hkv, int32_t group,
                                                     int32_t kv_chunk, int32_t zero_unseen,
                                                     uint32_t* __restrict__ kv_cnt, int64_t n_cnt) {
  tc::grid_launch_dependents();     // the KV kernel waits for this one where it reads D or the zeroed rows
  constexpr int LPR = D / 8;        // lanes per row (16 bytes each)
  constexpr int RPL = 32 / LPR;     // rows per warp load
  constexpr int RPW = 4 * RPL;      // rows per warp pass
  const int lane = threadIdx.x & 31;
  const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
  const int64_t n_pass = (n_rows + RPW - 1) / RPW;
  // When a pass's RPW rows are heads of one token (Hq a multiple of RPW) the
  // token is found with one 32-bit division a pass and a padding token's rows
  // are not read at all.
  const bool tok_pass = hq % RPW == 0 && n_rows < (int64_t(1) << 31);
  for (int64_t ps = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; ps < n_pass; ps += warps) {
    int pb = 0, pi = 0, ph = 0;
    bool live = true;
    if (tok_pass) {
      const uint32_t r0 = uint32_t(ps * RPW), tok = r0 / uint32_t(hq);
      pb = int(tok / uint32_t(t_pad));
      pi = int(tok - uint32_t(pb) * uint32_t(t_pad));
      ph = int(r0 - tok * uint32_t(hq));
      live = pi < n_tokens[pb];
    }
    uint4 va[4], vc[4];
    int64_t row[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      row[k] = ps * RPW + k * RPL + lane / LPR;
      va[k] = make_uint4(0, 0, 0, 0);
      vc[k] = va[k];
      if (row[k] < n_rows && live) {
        va[k] = reinterpret_cast<const uint4*>(o + row[k] * D)[lane % LPR];
        vc[k] = reinterpret_cast<const uint4*>(dout + row[k] * D)[lane % LPR];
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t a[4] = {va[k].x, va[k].y, va[k].z, va[k].w};
      const uint32_t c[4] = {vc[k].x, vc[k].y, vc[k].z, vc[k].w};
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        s += __uint_as_float(a[e] << 16) * __uint_as_float(c[e] << 16) +
             __uint_as_float(a[e] & 0xffff0000u) * __uint_as_float(c[e] & 0xffff0000u);
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (lane % LPR == 0 && row[k] < n_rows) {
        if (tok_pass) {
          const int h = ph + k * RPL + lane / LPR;
          dvec[(int64_t(pb) * hq + h) * t_pad + pi] = live ? s : 0.f;
        } else {
          const int h = int(row[k] % hq);
          const int64_t bt = row[k] / hq;
          const int b = int(bt / t_pad), i = int(bt % t_pad);
          dvec[(int64_t(b) * hq + h) * t_pad + i] = (i < n_tokens[b]) ? s : 0.f;
        }
      }
    }
  }
  for (int64_t x = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; x < n_cnt; x += int64_t(gridDim.x) * blockDim.x)
    kv_cnt[x] = 0u;  // bf16 gradients: per-warp item counters of split columns
  if (dk == nullptr) return;
  // zero the rows of split key columns (and with zero_unseen those of key
  // tiles no query sees): one (tree, key tile) unit per block pass
  const int64_t per_tile4 = int64_t(kB) * hkv * D / 4;  // float4s of one key tile's rows
  for (int u = blockIdx.x; u < n_trees * n_blk; u += gridDim.x) {
    const int b = u / n_blk, kb = u % n_blk;
    const int32_t* kp = k_ptr + b * (n_blk + 1);
    const int n_col = kp[kb + 1] - kp[kb];
    if (n_col == 0 ? !zero_unseen : group * n_col <= kv_chunk) continue;  // written whole by one item
    const int64_t base = (int64_t(b) * t_pad + int64_t(kb) * kB) * hkv * D / 4;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t x = threadIdx.x; x < per_tile4; x += blockDim.x) {
      dk[base + x] = z;
      dv[base + x] = z;
    }
  }
}

inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

int num_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 148;
  }
  return sms;
}

// Workspace of the backward: D [B, Hq, T] fp32, and for bf16 gradients the
// fp32 staging rows of split key columns (dK, dV: [B, T, Hkv, d] each) and the
// per-warp item counters [B, Hkv, T/128, 16].
struct BwdWs {
  uint64_t d, stage_k, stage_v, cnt, n_cnt, total;
};

BwdWs bwd_ws_layout(int64_t n_trees, int64_t t_pad, int64_t hq, int64_t hkv, int64_t d, bool f32) {
  BwdWs L{};
  uint64_t o = 0;
  L.d = o;
  o = align256(o + uint64_t(n_trees * hq * t_pad) * 4);
  if (!f32) {
    const uint64_t rows = uint64_t(n_trees * t_pad * hkv * d) * 4;
    L.stage_k = o;
    o = align256(o + rows);
    L.stage_v = o;
    o = align256(o + rows);
    L.cnt = o;
    L.n_cnt = uint64_t(n_trees * hkv * ((t_pad + kB - 1) / kB) * 4 * kNWG);
    o = align256(o + L.n_cnt * 4);
  }
  L.total = o;
  return L;
}

// Steps per KV work item: a quarter of one SM's share of the (query head,
// query tile) steps, estimated from the ancestor pairs (a full tile holds
// 128 x 128 of them), and at least kKvChunkMin, so that the longest key
// columns (the shared prefixes') are split just enough for the items to
// balance over the SMs.
int kv_chunk_for(const tpa_tree_view* tree, int hq, int group, int n_blk, int sms) {
  const int64_t est_steps = tree->ancestor_pairs * hq / (int64_t(kB) * kB);
  int64_t chunk = est_steps / (int64_t(sms) * 4);
  if (chunk < kKvChunkMin) chunk = kKvChunkMin;
  if (chunk > int64_t(group) * n_blk) chunk = int64_t(group) * n_blk;
  return int(chunk);
}

template <int D, bool F32OUT>
int launch_bwd(const tpa_tree_view* tree, const tpa_blockmask_view* mask, const void* q, const void* k,
               const void* v, const void* o, const float* lse, const void* dout, void* dq, void* dk,
               void* dv, void* ws, int hq, int hkv, float scale, cudaStream_t st) {
  const int64_t rows = int64_t(tree->n_trees) * tree->t_pad;
  const BwdWs L = bwd_ws_layout(tree->n_trees, tree->t_pad, hq, hkv, D, F32OUT);
  uint8_t* wsb = static_cast<uint8_t*>(ws);
  float* dvec = reinterpret_cast<float*>(wsb + L.d);
  float* stage_k = F32OUT ? nullptr : reinterpret_cast<float*>(wsb + L.stage_k);
  float* stage_v = F32OUT ? nullptr : reinterpret_cast<float*>(wsb + L.stage_v);
  uint32_t* kv_cnt = F32OUT ? nullptr : reinterpret_cast<uint32_t*>(wsb + L.cnt);
  const int64_t n_rows = rows * hq;
  const int G = hq / hkv;
  const int kv_chunk = kv_chunk_for(tree, hq, G, mask->n_blk, num_sms());
  bwd_pre_kernel<D><<<num_sms() * 8, 256, 0, st>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), tree->n_tokens,
      tree->t_pad, hq, n_rows, dvec, static_cast<float4*>(F32OUT ? dk : static_cast<void*>(stage_k)),
      static_cast<float4*>(F32OUT ? dv : static_cast<void*>(stage_v)), mask->k_ptr, tree->n_trees, mask->n_blk,
      hkv, G, kv_chunk, F32OUT ? 1 : 0, kv_cnt, int64_t(L.n_cnt));
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
  prm.sched = mask->sched;
  prm.stage_k = stage_k;
  prm.stage_v = stage_v;
  prm.kv_cnt = kv_cnt;
  prm.t_pad = tree->t_pad;
  prm.n_blk = mask->n_blk;
  prm.cap = mask->cap;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.kv_chunk = kv_chunk;
  prm.kv_nchunk = (G * mask->n_blk + prm.kv_chunk - 1) / prm.kv_chunk;
  prm.n_trees = tree->n_trees;
  prm.wide = ((reinterpret_cast<uintptr_t>(dq) | reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 31) == 0;
  prm.kv_items = tree->n_trees * hkv * mask->n_blk * prm.kv_nchunk;
  prm.dq_items = tree->n_trees * hq * mask->n_blk;
  prm.scale = scale;
  prm.scale_log2 = scale * kLog2e;
  const int sms = num_sms();
  TPA_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_kv_kernel<D, F32OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    KvCfg<D>::BYTES));
  {  // may start while the preprocess finishes (it waits where it needs its results)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(prm.kv_items < sms ? prm.kv_items : sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = KvCfg<D>::BYTES;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    TPA_CUDA_TRY(cudaLaunchKernelEx(&cfg, attn_bwd_kv_kernel<D, F32OUT>, tq, tk, tv, tdo, prm));
  }
  if constexpr (D == 128) {
    if (G % 2 == 0 && sms >= 2) {  // head pairs of one key/value head on the two SMs of a TPC
      CUtensorMap tk64, tv64;
      if (!tmap::make_rows_heads_d(&tk64, k, rows, hkv, D, 64) || !tmap::make_rows_heads_d(&tv64, v, rows, hkv, D, 64))
        return TPA_ERR_CUDA;
      prm.dq_items = tree->n_trees * (hq / 2) * mask->n_blk;
      const int pairs = prm.dq_items < sms / 2 ? prm.dq_items : sms / 2;
      TPA_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_dq2_kernel<D, F32OUT>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, Dq2Cfg<D>::BYTES));
      // starts on the SMs the KV kernel's last CTAs free (the two are independent)
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * pairs);
      cfg.blockDim = dim3(kThreads2);
      cfg.dynamicSmemBytes = Dq2Cfg<D>::BYTES;
      cfg.stream = st;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      TPA_CUDA_TRY(cudaLaunchKernelEx(&cfg, attn_bwd_dq2_kernel<D, F32OUT>, tq, tk64, tv64, tdo, prm));
      return TPA_OK;
    }
  }
  TPA_CUDA_TRY(cudaFuncSetAttribute(attn_bwd_dq_kernel<D, F32OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    DqCfg<D>::BYTES));
  attn_bwd_dq_kernel<D, F32OUT><<<prm.dq_items < sms ? prm.dq_items : sms, kThreads, DqCfg<D>::BYTES, st>>>(
      tq, tk, tv, tdo, prm);
  TPA_CUDA_TRY(cudaGetLastError());
  return TPA_OK;
}

}  // namespace

TPA_DEFINE_STATUS_READER(tpa_internal_status_bwd, g_status_bwd)

extern "C" uint64_t tpa_tree_attn_bwd_workspace_bytes(int32_t n_trees, int32_t t_pad, int32_t n_heads_q,
                                                      int32_t n_heads_kv, int32_t head_dim, int32_t grad_dtype) {
  if (n_trees < 1 || t_pad < 1 || n_heads_q < 1 || n_heads_kv < 1 || head_dim < 1) return 0;
  if (grad_dtype != TPA_GRAD_F32 && grad_dtype != TPA_GRAD_BF16) return 0;
  return bwd_ws_layout(n_trees, t_pad, n_heads_q, n_heads_kv, head_dim, grad_dtype == TPA_GRAD_F32).total;
}

extern "C" int tpa_tree_attn_bwd(const tpa_tree_view* tree, const tpa_blockmask_view* mask, const void* q,
                                 const void* k, const void* v, const void* o, const float* lse,
                                 const void* dout, void* dq, void* dk, void* dv, void* workspace,
                                 uint64_t workspace_bytes, int32_t n_heads_q, int32_t n_heads_kv,
                                 int32_t head_dim, float softmax_scale, int32_t grad_dtype, void* stream) {
  TPA_NVTX_RANGE("tpa_tree_attn_bwd");
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
      tpa_tree_attn_bwd_workspace_bytes(tree->n_trees, tree->t_pad, n_heads_q, n_heads_kv, head_dim, grad_dtype))
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
  TPA_NVTX_RANGE("tpa_tree_attn_bwd_noalloc");
  if (!tree) return TPA_ERR_INVALID_ARG;
  const uint64_t need = tpa_tree_attn_bwd_workspace_bytes(tree->n_trees, tree->t_pad, n_heads_q, n_heads_kv,
                                                         head_dim, grad_dtype);
  if (need == 0) return TPA_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return TPA_ERR_BUFFER_TOO_SMALL;
  void* scratch = nullptr;
  const int rc = noalloc_scratch(&scratch);
  if (rc != TPA_OK) return rc;
  return tpa_tree_attn_bwd(tree, mask, q, k, v, o, lse, dout, dq, dk, dv, scratch, kNoAllocScratchBytes,
                           n_heads_q, n_heads_kv, head_dim, softmax_scale, grad_dtype, stream);
}
