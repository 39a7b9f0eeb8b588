// Tree attention forward on tcgen05 tensor cores (sm_103a).
//
// Semantics (tree training page, §树构建过程 mask caption, §注意力机制): query
// i of a packed tree sees key j iff j <= i <= E[j] (j is i or an ancestor);
// O_i = softmax over the visible keys of scale * q_i.k_j, times v_j.
// Only non-empty 128x128 tiles are visited (the per-query-block CSR of the
// classifier); PARTIAL tiles apply the precomputed 128-bit row masks, FULL
// tiles apply nothing.
//
// Persistent kernel: one CTA per SM takes work items from a global counter
// (heaviest first; one 128-query tile of
// NH query heads that share a key/value head, NH = 2 when the group size
// allows it), so K/V tiles are loaded once for both heads and the mask is
// shared, and one item's fill and drain (Q load, first S, O epilogue) overlap
// its neighbours'.  Barrier phases run on across items.  Warp roles:
//   warpgroup h < NH  softmax of head h: thread r owns query row r (TMEM lane
//                     r); fp32 online softmax in the log2 domain with packed
//                     f32x2 arithmetic; P (bf16) goes to TMEM over the S
//                     columns it replaces and feeds the TS-form PV MMA;
//                     O is rescaled in TMEM only when the running max grows
//                     by more than 2^8 (exact: numerator and denominator keep
//                     the same stale max).
//   warp 4*NH         TMA producer (one thread): Q of each item, then K and V
//                     tiles through separate rings.
//   warp 4*NH+1       MMA issuer (one thread).  Per key tile j and head h:
//                     PV_h(j) then S_h(j+1), so head B's softmax runs while
//                     head A's MMAs run (ping-pong) and the tensor core always
//                     has the other head's work queued.
// TMEM columns: S_h [128h, 128h+128) (P_h aliased on its first 64 columns),
// O_h [128 NH + 128h, ...).  O / l leaves through a 16 KB swizzled shared-
// memory stage per head and bulk tensor stores.
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
  const int32_t* q_ptr;
  const int32_t* q_idx;
  const uint4* qmask;
  uint32_t* sched;   // [0] next work item, [1] finished CTAs (both back to 0 at kernel end)
  int32_t t_pad, n_blk, cap, hq, hkv, n_items;
  int32_t wide;      // o is 32-byte aligned: its rows go out 32 bytes at a time
  float scale_log2;  // softmax scale * log2(e)
};

template <int D, int NH>
struct FwdCfg {
  static constexpr int NCH = D / 64;
  static constexpr uint32_t TILE = NCH * kChunk;   // one 128 x D bf16 tile
  // O leaves through the TMA engine, 64 columns (one 16 KB swizzled box) of
  // a head at a time, staged here per head
  static constexpr uint32_t STAGE = NH * kChunk;
  static constexpr uint32_t BASE = NH * TILE + STAGE + 512;  // + barriers and flags
  static constexpr int NS_FIT = int((kSmemMax - 1024 - BASE) / (2 * TILE));
  static constexpr int NS = NS_FIT > 3 ? 3 : NS_FIT;  // K and V ring depth
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NH * TILE;
  static constexpr uint32_t OFF_V = OFF_K + NS * TILE;
  static constexpr uint32_t OFF_STAGE = OFF_V + NS * TILE;
  static constexpr uint32_t OFF_BAR = OFF_STAGE + STAGE;
  // q_full, q_empty, k_full[NS], k_empty[NS], v_full[NS], v_empty[NS], s_full[NH], p_full[NH],
  // o_free[NH], stage_full[NH], stage_free[NH], o_final, drain, item_full[2], item_empty[2]
  static constexpr int NBAR = 2 + 4 * NS + 5 * NH + 2 + 4;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t BYTES = OFF_MISC + 32 + 1024;  // + alignment slack
  // Two heads: three full warpgroups (the third holds the TMA and MMA warps and
  // two idle ones) so that registers can move between warpgroups: launched at
  // REG_LAUNCH a thread, the producer/issuer warpgroup drops to REG_LOW and the
  // softmax warpgroups rise to REG_HIGH, within what the CTA was launched with
  // (at 168 the softmax spilled; its code fits in 184 and the producer's and
  // issuer's in 120).
  static constexpr int THREADS = NH == 2 ? 384 : 128 * NH + 64;
  static constexpr int REG_LAUNCH = 168, REG_LOW = 120, REG_HIGH = 184;
  static_assert(NH != 2 || REG_HIGH * 256 + REG_LOW * 128 <= REG_LAUNCH * 384, "register split");
  static constexpr uint32_t TMEM_COLS = NH == 2 ? 512 : 256;
  static_assert(NS >= 1, "shared memory too small");
  static_assert(BYTES <= kSmemMax, "shared memory budget");
};

using tc::add2;
using tc::f2;
using tc::fma2;
using tc::unf2;
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

// Work item -> (tree, first query head, query block); deepest blocks first.
struct Item {
  int b, h0, qb, e0, n_it;
};
template <int NH>
__device__ __forceinline__ Item decode_item(const FwdParams& p, int it) {
  Item r;
  const int per_tree = p.n_blk * (p.hq / NH);
  r.b = it / per_tree;
  const int rem = it - r.b * per_tree;
  r.h0 = (rem / p.n_blk) * NH;
  r.qb = p.n_blk - 1 - rem % p.n_blk;
  const int32_t* rp = p.q_ptr + r.b * (p.n_blk + 1);
  r.e0 = rp[r.qb];
  r.n_it = rp[r.qb + 1] - r.e0;
  return r;
}

template <int D, int NH>
__global__ void __launch_bounds__(FwdCfg<D, NH>::THREADS, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const FwdParams p) {
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
  uint64_t* q_empty = bar + 1;
  uint64_t* k_full = bar + 2;
  uint64_t* k_empty = k_full + NS;
  uint64_t* v_full = k_empty + NS;
  uint64_t* v_empty = v_full + NS;
  uint64_t* s_full = v_empty + NS;
  uint64_t* p_full = s_full + NH;
  uint64_t* o_free = p_full + NH;
  uint64_t* stage_full = o_free + NH;     // [NH]: the warpgroup wrote its O stage
  uint64_t* stage_free = stage_full + NH;  // [NH]: the TMA engine has read it
  uint64_t* o_final = stage_free + NH;
  uint64_t* drain = o_final + 1;
  uint64_t* item_full = drain + 1;   // [2]
  uint64_t* item_empty = drain + 3;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* item_ring = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);  // [2]

  const int warp = threadIdx.x >> 5;
  const int hkv_group = p.hq / p.hkv;
  constexpr int W_TMA = 4 * NH, W_MMA = 4 * NH + 1;

  if (threadIdx.x == 0) {
    tc::mbar_init(q_full, 1);
    tc::mbar_init(q_empty, 1);
    for (int s = 0; s < NS; ++s) {
      tc::mbar_init(k_full + s, 1);
      tc::mbar_init(k_empty + s, 1);
      tc::mbar_init(v_full + s, 1);
      tc::mbar_init(v_empty + s, 1);
    }
    for (int h = 0; h < NH; ++h) {
      tc::mbar_init(s_full + h, 1);
      tc::mbar_init(p_full + h, 128);
      tc::mbar_init(o_free + h, 128);
      tc::mbar_init(stage_full + h, 128);
      tc::mbar_init(stage_free + h, 1);
    }
    tc::mbar_init(o_final, 1);
    tc::mbar_init(drain, 1);
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(item_full + s, 1);
      tc::mbar_init(item_empty + s, 1 + 128 * NH);
    }
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == W_MMA) tc::tmem_alloc(tmem_slot, C::TMEM_COLS);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= W_TMA) {
  // the producer/issuer warpgroup gives registers to the softmax warpgroups
  // (all four of its warps execute this; two of them have no role)
  if constexpr (NH == 2) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_LOW));
  if (warp == W_TMA) {
    // ------------------------------------------------------------ producer
    // One thread runs the whole loop, like the MMA issuer: a warp-level sync
    // right after the bulk copies would hold the warp until they are issued.
    if (tc::elect_one()) {
      tc::tma_prefetch_desc(&tm_q);
      tc::tma_prefetch_desc(&tm_k);
      tc::tma_prefetch_desc(&tm_v);
      auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_fwd); };
      int kt = 0, vt = 0, nq = 0;  // ring counters and non-empty items so far
      bool ok = true;
      for (int k = 0; ok; ++k) {
        // fetch the next work item and hand it to the other roles
        if (!(ok = wait1(item_empty + (k & 1), ((k >> 1) & 1) ^ 1))) break;
        const uint32_t u = atomicAdd(p.sched, 1u);
        const int it = u < uint32_t(p.n_items) ? int(u) : -1;  // unsigned: no index below 0
        item_ring[k & 1] = it;
        tc::mbar_arrive(item_full + (k & 1));
        if (it < 0) break;
        const Item I = decode_item<NH>(p, it);
        if (I.n_it == 0) continue;
        const int32_t* list = p.q_idx + int64_t(I.b) * p.cap + I.e0;
        const int g = I.h0 / hkv_group;
        if (!(ok = wait1(q_empty, (nq & 1) ^ 1))) break;
        tc::mbar_arrive_expect_tx(q_full, NH * TILE);
        for (int h = 0; h < NH; ++h)
          for (int c = 0; c < NCH; ++c)
            tc::tma_load_3d(sQ + h * TILE + c * kChunk, &tm_q, q_full, c * 64, I.h0 + h, I.b * p.t_pad + I.qb * kB);
        // K runs ahead of V by one tile: the MMA needs K(j+1) before V(j).
        int kj = 0, vj = 0;
        while (kj < I.n_it || vj < I.n_it) {
          const bool do_k = kj < I.n_it && kj <= vj + 1;
          const int j = do_k ? kj : vj;
          const int krow = I.b * p.t_pad + (list[j] >> 1) * kB;
          const int gx = (do_k ? kt : vt) + j, s = gx % NS;
          if (!(ok = wait1((do_k ? k_empty : v_empty) + s, ((gx / NS) & 1) ^ 1))) break;
          uint64_t* fb = (do_k ? k_full : v_full) + s;
          uint8_t* dst = (do_k ? sK : sV) + s * TILE;
          tc::mbar_arrive_expect_tx(fb, TILE);
          for (int c = 0; c < NCH; ++c)
            tc::tma_load_3d(dst + c * kChunk, do_k ? &tm_k : &tm_v, fb, c * 64, g, krow);
          if (do_k) ++kj; else ++vj;
        }
        kt += kj;
        vt += vj;
        ++nq;
      }
      if (*abort_flag) {  // let the copies already issued land before the CTA exits
        volatile int never = 0;
        for (int j = (kt > NS ? kt - NS : 0); j < kt; ++j)
          tc::mbar_wait(k_full + (j % NS), (j / NS) & 1, &never, &g_status_fwd, 100000000ull);
        for (int j = (vt > NS ? vt - NS : 0); j < vt; ++j)
          tc::mbar_wait(v_full + (j % NS), (j / NS) & 1, &never, &g_status_fwd, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    // One thread runs the whole loop.  A warp-level sync after tcgen05.mma
    // holds the warp until the thread's queued MMAs have gone into the pipe,
    // so with the warp in step every wait between MMA groups would leave the
    // tensor pipe idle; a lone thread's waits overlap the queued MMAs.
    constexpr uint32_t idesc_qk = tc::idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_pv = tc::idesc_bf16(128, D, false, true);
    // Descriptors are built once; a k-step or stage only adds (byte offset >> 4)
    // to the 14-bit start-address field (shared addresses stay below 2^18).
    const uint64_t dQ = tc::smem_desc(tc::smem_u32(sQ), 16, 1024);
    const uint64_t dK = tc::smem_desc(tc::smem_u32(sK), 16, 1024);
    const uint64_t dV = tc::smem_desc(tc::smem_u32(sV), kChunk, 1024);
    auto issue_s = [&](int h, int s) {  // S_h = Q_h K(s)^T
      const uint64_t qa = dQ + ((h * TILE) >> 4), kb_ = dK + ((s * TILE) >> 4);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = ((k >> 2) * kChunk + (k & 3) * 32) >> 4;
        tc::mma_ss(tmem + h * 128, qa + off, kb_ + off, idesc_qk, k > 0);
      }
      tc::mma_commit(s_full + h);
    };
    auto issue_pv = [&](int h, int s, bool first) {  // O_h (+)= P_h V(s), P_h read from TMEM
      const uint64_t vb = dV + ((s * TILE) >> 4);
#pragma unroll
      for (int k = 0; k < kB / 16; ++k)
        mma_ts(tmem + 128 * NH + h * 128, tmem + h * 128 + k * 8, vb + ((k * 2048) >> 4), idesc_pv,
               (!first || k > 0) ? 1u : 0u);
    };
    auto commit = [&](uint64_t* b_) { tc::mma_commit(b_); };
    auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_fwd); };
    if (tc::elect_one()) {
    int kt = 0, vt = 0, tb = 0, nq = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!(ok = wait1(item_full + (k & 1), (k >> 1) & 1))) break;
      const int it = item_ring[k & 1];
      tc::mbar_arrive(item_empty + (k & 1));
      if (it < 0) break;
      const Item I = decode_item<NH>(p, it);
      const int n_it = I.n_it;
      if (n_it == 0) continue;
      // S_h(0): the S regions were last read by the previous item's PV (issued
      // earlier, executed in order) and its softmax (done before its p_full).
      if (!(ok = wait1(q_full, nq & 1) && wait1(k_full + kt % NS, (kt / NS) & 1))) break;
      tc::tc_fence_after();
      for (int h = 0; h < NH; ++h) issue_s(h, kt % NS);
      commit(k_empty + kt % NS);
      if (n_it == 1) commit(q_empty);
      for (int j = 0; ok && j < n_it; ++j) {
        const int gv = vt + j, sv = gv % NS;
        const int gk1 = kt + j + 1, s1 = gk1 % NS;
        const bool more = j + 1 < n_it;
        if (!(ok = wait1(v_full + sv, (gv / NS) & 1))) break;
        for (int h = 0; h < NH && ok; ++h) {
          if (!(ok = wait1(p_full + h, (tb + j) & 1))) break;
          if (j == 0 && nq > 0 && !(ok = wait1(o_free + h, (nq - 1) & 1))) break;
          tc::tc_fence_after();
          issue_pv(h, sv, j == 0);
          if (more) {
            if (h == 0 && !(ok = wait1(k_full + s1, (gk1 / NS) & 1))) break;
            tc::tc_fence_after();
            issue_s(h, s1);
          }
        }
        if (!ok) break;
        commit(v_empty + sv);
        if (more) {
          commit(k_empty + s1);
          if (j + 2 == n_it) commit(q_empty);  // the item's last S was just issued
        }
      }
      if (ok) commit(o_final);
      kt += n_it;
      vt += n_it;
      tb += n_it;
      ++nq;
    }
    if (*abort_flag) {  // let issued MMAs finish before TMEM is released
      volatile int never = 0;
      tc::mma_commit(drain);
      tc::mbar_wait(drain, 0, &never, &g_status_fwd, 100000000ull);
    }
    }
    __syncwarp();
  }
  } else {
    if constexpr (NH == 2) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_HIGH));
    // ------------------------------------------------------------ softmax (head h)
    const int h = warp >> 2;
    const int r = threadIdx.x & 127;   // query row within the tile = TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + h * 128;
    const uint32_t tO = tmem + lane_base + 128 * NH + h * 128;
    const uint64_t sl2 = f2(p.scale_log2, p.scale_log2);
    auto wait_all = [&](uint64_t* b_, uint32_t par) {
      return __all_sync(0xffffffffu, tc::mbar_wait(b_, par, abort_flag, &g_status_fwd));
    };
    int tb = 0, nq = 0;
    int su = 0;  // uses of this warpgroup's O stage so far
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!wait_all(item_full + (k & 1), (k >> 1) & 1)) break;
      const int it = item_ring[k & 1];
      tc::mbar_arrive(item_empty + (k & 1));
      if (it < 0) break;
      const Item I = decode_item<NH>(p, it);
      const int n_it = I.n_it;
      const int row0 = I.b * p.t_pad + I.qb * kB;
      const int i = I.qb * kB + r;     // query position in the tree
      __nv_bfloat16* orow = p.o + (int64_t(row0 + r) * p.hq + I.h0 + h) * D;
      float* lse_out = p.lse + (int64_t(I.b) * p.hq + I.h0 + h) * p.t_pad + i;
      if (n_it == 0) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = z;
        *lse_out = 0.f;
        continue;
      }
      const int32_t* list = p.q_idx + int64_t(I.b) * p.cap + I.e0;
      const uint4* qmask_row = p.qmask + (int64_t(I.b) * p.cap + I.e0) * kB + r;
      float m_run = -INFINITY, l_run = 0.f;
      int entry = list[0];
      uint4 mk = (entry & 1) ? make_uint4(0, 0, 0, 0) : qmask_row[0];
      for (int j = 0; j < n_it; ++j) {
        const bool full = entry & 1;
        const uint4 mcur = mk;
        if (j + 1 < n_it) {  // prefetch the next tile's entry and mask row
          entry = list[j + 1];
          if (!(entry & 1)) mk = qmask_row[int64_t(j + 1) * kB];
        }
        if (!wait_all(s_full + h, (tb + j) & 1)) { ok = false; break; }
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
        // row max: 8 independent chains, then a short tree
        float mxs[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) mxs[t] = fmaxf(__uint_as_float(sv[2 * t]), __uint_as_float(sv[2 * t + 1]));
#pragma unroll
        for (int c = 16; c < 128; c += 16)
#pragma unroll
          for (int t = 0; t < 8; ++t)
            mxs[t] = max3(mxs[t], __uint_as_float(sv[c + 2 * t]), __uint_as_float(sv[c + 2 * t + 1]));
        const float mx = fmaxf(max3(mxs[0], mxs[1], mxs[2]), max3(mxs[3], mxs[4], max3(mxs[5], mxs[6], mxs[7])));
        const float m_new = fmaxf(m_run, mx * p.scale_log2);
        const bool resc = m_new > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
          alpha = tc::ex2(m_run - m_new);
          m_run = m_new;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        const uint64_t negm = f2(-m_use, -m_use);
        uint64_t sum2[4] = {f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f), f2(0.f, 0.f)};  // 4 chains
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float a, bb;
          unf2(fma2(f2(__uint_as_float(sv[2 * c]), __uint_as_float(sv[2 * c + 1])), sl2, negm), a, bb);
          const float p0 = tc::ex2(a), p1 = tc::ex2(bb);
          sum2[c & 3] = add2(sum2[c & 3], f2(p0, p1));
          pk[c] = tc::pack_bf16(p0, p1);
        }
        float s_lo, s_hi;
        unf2(add2(add2(sum2[0], sum2[1]), add2(sum2[2], sum2[3])), s_lo, s_hi);
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
      if (!ok || !wait_all(o_final, nq & 1)) { ok = false; break; }
      tc::tc_fence_after();
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      // O_h / l as bf16 through a 16 KB swizzled stage, 64 columns at a time,
      // written out by the TMA engine: the item's 32 KB of O rows do not hold
      // up this warpgroup's next loads and barrier waits behind a burst of
      // stores.  Thread r == 0 issues the copies; before a refill it waits
      // until the engine has read the stage and frees it for the others.
      uint8_t* stg = smem + C::OFF_STAGE + h * kChunk;
      const int orow0 = I.b * p.t_pad + I.qb * kB;
      for (int half = 0; half < NCH && ok; ++half, ++su) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t ov[32];
          tc::tmem_ld32(tO + half * 64 + c * 32, ov);
          tc::tmem_ld_wait();
#pragma unroll
          for (int u = 0; u < 16; ++u)
            w[16 * c + u] = tc::pack_bf16(__uint_as_float(ov[2 * u]) * inv, __uint_as_float(ov[2 * u + 1]) * inv);
        }
        if (half == NCH - 1) {
          tc::tc_fence_before();
          tc::mbar_arrive(o_free + h);  // O_h may be overwritten by the next item
        }
        if (su > 0) {
          if (r == 0) {
            tc::bulk_wait_read();
            tc::mbar_arrive(stage_free + h);
          }
          if (!wait_all(stage_free + h, (su - 1) & 1)) { ok = false; break; }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(stg + tc::sw128_offset(uint32_t(r), uint32_t(c))) =
              make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(stage_full + h);
        bool staged = true;
        if (r == 0) {
          staged = tc::mbar_wait(stage_full + h, su & 1, abort_flag, &g_status_fwd);
          if (staged) {
            tc::tma_store_3d(&tm_o, stg, half * 64, I.h0 + h, orow0);
            tc::bulk_commit();
          }
        }
        if (!__all_sync(0xffffffffu, staged)) { ok = false; break; }
      }
      if (!ok) break;
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      *lse_out = l_run > 0.f ? (m_use + __log2f(l_run)) * kLn2 : 0.f;
      tb += n_it;
      ++nq;
    }
  }

  if (warp < W_TMA && (threadIdx.x & 127) == 0) tc::bulk_wait_all();  // this warpgroup's O copies
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == W_MMA) tc::tmem_dealloc(tmem, C::TMEM_COLS);
  if (threadIdx.x == 0) {  // the last CTA to finish rearms the work counter for the next call
    __threadfence();
    if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
      p.sched[0] = 0;
      p.sched[1] = 0;
      __threadfence();
    }
  }
}

int num_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 148;
  }
  return sms;
}

// launch_fwd_cfg<D, 2> returns this (not a library status) when the two-head
// kernel was not compiled to the register count its setmaxnreg split assumes
constexpr int kFwdRegsMismatch = 1;

template <int D, int NH>
int launch_fwd_cfg(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                   FwdParams prm,
                   int n_trees, cudaStream_t st) {
  using C = FwdCfg<D, NH>;
  prm.n_items = prm.n_blk * (prm.hq / NH) * n_trees;
  const int grid = prm.n_items < num_sms() ? prm.n_items : num_sms();
  TPA_CUDA_TRY(cudaFuncSetAttribute(attn_fwd_kernel<D, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::BYTES));
  if constexpr (NH == 2) {
    // setmaxnreg.inc waits until the warpgroups' registers fit in what the CTA was
    // launched with: launch only when the kernel was compiled to REG_LAUNCH a thread
    // (the caller then runs the one-head kernel instead)
    cudaFuncAttributes fa;
    TPA_CUDA_TRY(cudaFuncGetAttributes(&fa, attn_fwd_kernel<D, NH>));
    if (fa.numRegs != C::REG_LAUNCH) return kFwdRegsMismatch;
  }
  attn_fwd_kernel<D, NH><<<grid, C::THREADS, C::BYTES, st>>>(tq, tk, tv, to, prm);
  TPA_CUDA_TRY(cudaGetLastError());
  return TPA_OK;
}

template <int D>
int launch_fwd(const tpa_tree_view* tree, const tpa_blockmask_view* mask, const void* q, const void* k,
               const void* v, void* o, float* lse, int hq, int hkv, float scale, cudaStream_t st) {
  const uint64_t rows = uint64_t(tree->n_trees) * tree->t_pad;
  CUtensorMap tq, tk, tv, to;
  if (!tmap::make_rows_heads_d(&tq, q, rows, hq, D) || !tmap::make_rows_heads_d(&tk, k, rows, hkv, D) ||
      !tmap::make_rows_heads_d(&tv, v, rows, hkv, D) || !tmap::make_rows_heads_d(&to, o, rows, hq, D))
    return TPA_ERR_CUDA;
  FwdParams prm;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.wide = (reinterpret_cast<uintptr_t>(o) & 31) == 0;
  prm.lse = lse;
  prm.q_ptr = mask->q_ptr;
  prm.q_idx = mask->q_idx;
  prm.qmask = reinterpret_cast<const uint4*>(mask->qmask);
  prm.sched = mask->sched;
  prm.t_pad = tree->t_pad;
  prm.n_blk = mask->n_blk;
  prm.cap = mask->cap;
  prm.hq = hq;
  prm.hkv = hkv;
  prm.n_items = 0;
  prm.scale_log2 = scale * kLog2e;
  if ((hq / hkv) % 2 == 0) {
    const int rc = launch_fwd_cfg<D, 2>(tq, tk, tv, to, prm, tree->n_trees, st);
    if (rc != kFwdRegsMismatch) return rc;
  }
  return launch_fwd_cfg<D, 1>(tq, tk, tv, to, prm, tree->n_trees, st);
}

// One thread waits on an mbarrier with the bounded wait every role of the
// attention kernels uses.  arrive != 0: the thread completes the phase itself
// first, so the wait succeeds; arrive == 0: nothing arrives, the wait gives up
// after about limit_ns, raises the abort flag and sets the device status word.
__global__ void wait_probe_kernel(uint64_t limit_ns, int arrive) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  tc::mbar_init(&bar, 1);
  tc::fence_mbar_init();
  if (arrive) tc::mbar_arrive(&bar);
  (void)tc::mbar_wait(&bar, 0, &abort_flag, &g_status_fwd, limit_ns);
}

}  // namespace

TPA_DEFINE_STATUS_READER(tpa_internal_status_fwd, g_status_fwd)

extern "C" int tpa_wait_probe(uint64_t limit_ns, int32_t arrive, void* stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return TPA_ERR_INVALID_ARG;
  wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, arrive);
  TPA_CUDA_TRY(cudaGetLastError());
  return TPA_OK;
}

int tpa_internal_check_attn_args(const tpa_tree_view* tree, const tpa_blockmask_view* mask, int hq,
                                 int hkv, int d) {
  if (!tree || !mask || !tree->subtree_end || !tree->n_tokens || !mask->q_ptr || !mask->q_idx ||
      !mask->k_ptr || !mask->k_idx || !mask->qmask || !mask->sched)
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
  TPA_NVTX_RANGE("tpa_tree_attn_fwd");
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
