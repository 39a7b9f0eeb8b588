// LM head fused into the log-probability pass (tree training page,
// §对数概率计算, with the step upstream of it folded in): the logits of tree
// row r are logits[r, v] = sum_k hidden[r, k] * weight[v, k]; they are formed
// tile by tile on tcgen05 tensor cores and consumed in place — online
// softmax statistics and the labels of the row — so they never reach HBM.
//
// Kernel 1 (lmh_kernel), persistent, on CTA pairs: the two CTAs of a
// cluster (the two SMs of a TPC) take a work item, a (256-row tile, chunk of
// kVt 256-wide vocab tiles) pair, CTA c holding rows [128c, 128c+128) of the
// tile; every MMA runs once over the pair with M = 256 (tcgen05
// cta_group::2), each CTA loading its own 128 hidden rows and half of the
// 256 weight rows of the vocab tile, so a weight tile crosses L2 once per 256
// rows (a third fewer bytes per FLOP than single-CTA 128-row tiles).  Items
// run in row groups so the hidden rows of a group stay in L2 while its vocab
// chunks stream past.  Roles (in each CTA):
//   warp 16        TMA producer: per vocab tile and 64-wide slice of H, the
//                  CTA's 128x64 hidden tile and 128x64 weight half-tile into
//                  a 6-stage ring (32 KB a stage); the even CTA takes the
//                  items and writes them into both CTAs' rings.
//   warp 17        MMA issuer (even CTA): tcgen05.mma kind::f16, M=256 N=256
//                  K=16, into one of two 256-column TMEM accumulators (each
//                  CTA's own 128 rows), so a tile's epilogue overlaps the
//                  next tile's MMAs.
//   warps 0-15     epilogue: thread r of warpgroup w reads columns
//                  [64w, 64w+64) of row r, keeps the row's running max m,
//                  s = sum exp(x - m) and t = sum exp(x - m) x over its
//                  columns, and stores the raw logit of every label of the row
//                  (the token of each child position) that falls in them.
//                  At the item's end the four warpgroups' (m, s, t) of a row
//                  are merged in shared memory into one partial per (row,
//                  chunk).
// Kernel 2 (lmh_combine_kernel): per tree position, merge the partials of its
// row into lse = M + log S and entropy = lse - T / S, and write
// pos_logp[c] = logit[c] - lse for each child c; then the per-sequence gather
// of the log-prob pass.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "device_common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "tmap.h"

namespace {

__device__ unsigned int g_status_lmh = 0;

constexpr int kBM = 128, kBN = 256, kBK = 64;      // kBM: rows of one CTA (a pair takes 2 kBM)
constexpr int kVt = 8;                               // vocab tiles per work item
constexpr int kStages = 6;
constexpr uint32_t kATile = kBM * kBK * 2;           // 16 KB: this CTA's hidden rows
constexpr uint32_t kBTile = kBN / 2 * kBK * 2;       // 16 KB: this CTA's half of the weight tile
constexpr uint32_t kStage = kATile + kBTile;
constexpr int kThreads = 576;                        // 16 epilogue warps + TMA + MMA
constexpr int kWTma = 16, kWMma = 17;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint32_t kOffMerge = kStages * kStage;     // [2 item parities][3 warpgroups][128 rows] (m, s, t, -)
constexpr uint32_t kOffBar = kOffMerge + 2 * 3 * kBM * 16;
// full[kStages], empty[kStages], acc_full[2], acc_free[2], item_full[2], item_empty[2], drain,
// merge_full[2], merge_free[2] (full, acc_free and item_empty are used on the even CTA)
constexpr int kNBar = 2 * kStages + 13;
constexpr uint32_t kOffMisc = kOffBar + kNBar * 8;
constexpr uint32_t kSmemBytes = kOffMisc + 32;       // base checked 1024-byte aligned
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct LmhParams {
  const int32_t* n_tokens;
  const int64_t* tok_base;
  const int32_t* tokens;
  const int32_t* child_off;
  const int32_t* child_pos;
  float4* part;        // [rows][n_vc] (m, s, t, -)
  float* pair_logit;   // [B*T_pad] raw logit of each position's token under its parent row
  uint32_t* ctr;       // work counter, zeroed before every launch
  int64_t rows;
  int32_t n_trees, t_pad, vocab, hidden, n_rt, n_vt, n_vc, group, n_items;
};

struct LmhItem {
  int rt, vc;
};

__device__ __forceinline__ LmhItem decode(const LmhParams& p, int it) {
  const int per_group = p.group * p.n_vc;
  const int g = it / per_group;
  const int base = g * p.group;
  const int rg = min(p.group, p.n_rt - base);
  const int rem = it - g * per_group;
  return LmhItem{base + rem % rg, rem / rg};
}

// one arrival per warp on the even CTA's copy of `bar`
__device__ __forceinline__ void warp_arrive_lead(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) tc::mbar_arrive_remote(tc::peer_addr(bar, 0));
  __syncwarp();
}

// Tree and position of compact row r (tok_base is the exclusive prefix sum).
__device__ __forceinline__ void row_to_pos(const LmhParams& p, int64_t r, int& b, int& pos) {
  int lo = 0, hi = p.n_trees - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.tok_base[mid] <= r) lo = mid; else hi = mid - 1;
  }
  b = lo;
  pos = int(r - p.tok_base[lo]);
}

struct Stats {
  float m, s, t;
};

__device__ __forceinline__ void stats_merge(Stats& a, const Stats& b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -INFINITY) return;
  const float ca = tc::ex2((a.m - m) * kLog2e), cb = tc::ex2((b.m - m) * kLog2e);
  a.s = a.s * ca + b.s * cb;
  a.t = a.t * ca + b.t * cb;
  a.m = m;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    lmh_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
               const LmhParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (tc::smem_u32(smem) & 1023u) {  // the same for every CTA of the launch: all leave
    if (threadIdx.x == 0) atomicOr(&g_status_lmh, 2u);
    return;
  }
  const uint32_t crank = tc::cta_rank();
  const bool lead = crank == 0;
  float4* sMerge = reinterpret_cast<float4*>(smem + kOffMerge);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint64_t* full = bar;
  uint64_t* empty = bar + kStages;
  uint64_t* acc_full = bar + 2 * kStages;     // [2]
  uint64_t* acc_free = acc_full + 2;          // [2]
  uint64_t* item_full = acc_full + 4;         // [2]
  uint64_t* item_empty = acc_full + 6;        // [2]
  uint64_t* drain = acc_full + 8;
  uint64_t* merge_full = acc_full + 9;        // [2]: warpgroups 1-3 have written an item's statistics
  uint64_t* merge_free = acc_full + 11;       // [2]: warpgroup 0 has read them
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  volatile int* item_ring = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);  // [2]
  const int warp = threadIdx.x >> 5;
  const int n_k = p.hidden / kBK;
  // item-slot consumers, on the even CTA: its MMA thread and 16 epilogue
  // warps, the odd CTA's producer and 16 epilogue warps
  constexpr int kCons = 1 + 16 + 1 + 16;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(full + s, 1);
      tc::mbar_init(empty + s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(acc_full + s, 1);
      tc::mbar_init(acc_free + s, 32);  // one arrival per epilogue warp of either CTA
      tc::mbar_init(item_full + s, 1);
      tc::mbar_init(item_empty + s, kCons);
      tc::mbar_init(merge_full + s, 384);
      tc::mbar_init(merge_free + s, 128);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == kWMma) tc::tmem_alloc2(tmem_slot, 512);
  tc::tc_fence_before();
  tc::cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto wait_u = [&](uint64_t* b_, uint32_t par) {
    return __all_sync(0xffffffffu, tc::mbar_wait(b_, par, abort_flag, &g_status_lmh));
  };
  auto wait_ring = [&](uint64_t* b_, uint32_t par) {  // item slots: written across the pair
    return __all_sync(0xffffffffu, tc::mbar_wait_cluster(b_, par, abort_flag, &g_status_lmh));
  };

  if (warp == kWTma) {
    // ------------------------------------------------------------ producer
    // The producer and the MMA issuer each run their whole loop on one elected
    // thread: a warp-level sync right after tcgen05.mma (or a bulk copy) holds
    // the warp until the queued operations have gone out, which would leave
    // the tensor pipe idle for the length of every wait between k-stages.
    if (tc::elect_one()) {
      tc::tma_prefetch_desc(&tm_h);
      tc::tma_prefetch_desc(&tm_w);
      auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_lmh); };
      int q = 0;  // stage loads issued
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int it;
        if (lead) {  // take the pair's next item, into both CTAs' rings
          if (!(ok = wait1(item_empty + (k & 1), ((k >> 1) & 1) ^ 1))) break;
          const uint32_t u = atomicAdd(p.ctr, 1u);
          it = u < uint32_t(p.n_items) ? int(u) : -1;
          item_ring[k & 1] = it;
          tc::st_cluster_u32(tc::peer_addr(const_cast<int*>(item_ring + (k & 1)), 1), uint32_t(it));
          tc::mbar_arrive(item_full + (k & 1));
          tc::mbar_arrive_release_cluster(tc::peer_addr(item_full + (k & 1), 1));  // after the ring store
        } else {
          if (!(ok = tc::mbar_wait_cluster(item_full + (k & 1), (k >> 1) & 1, abort_flag, &g_status_lmh))) break;
          it = item_ring[k & 1];
          tc::mbar_arrive_remote(tc::peer_addr(item_empty + (k & 1), 0));
        }
        if (it < 0) break;
        const LmhItem I = decode(p, it);
        const int vt1 = min(p.n_vt, (I.vc + 1) * kVt);
        const int rows0 = I.rt * 2 * kBM + kBM * int(crank);  // this CTA's hidden rows
        for (int vt = I.vc * kVt; ok && vt < vt1; ++vt) {
          for (int kc = 0; kc < n_k; ++kc, ++q) {
            const int s = q % kStages;
            if (!(ok = wait1(empty + s, ((q / kStages) & 1) ^ 1))) break;
            uint8_t* dst = smem + s * kStage;
            if (lead) tc::mbar_arrive_expect_tx(full + s, 2 * kStage);  // both CTAs' tiles
            const uint32_t lb = tc::peer_addr(full + s, 0);
            tc::tma_load_3d_pair(dst, &tm_h, lb, kc * kBK, 0, rows0);
            tc::tma_load_3d_pair(dst + kATile, &tm_w, lb, kc * kBK, 0, vt * kBN + kBN / 2 * int(crank));
          }
        }
      }
      if (*abort_flag) {  // copies into this CTA's shared memory complete on the even CTA's barriers:
        const long long t0 = clock64();  // give any still in flight time to land before the CTA leaves
        while (clock64() - t0 < 400000) {
        }
      }
    }
    __syncwarp();
  } else if (warp == kWMma) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = tc::idesc_bf16(2 * kBM, kBN, false, false);
    const uint64_t dA = tc::smem_desc(tc::smem_u32(smem), 16, 1024);
    const uint64_t dB = tc::smem_desc(tc::smem_u32(smem + kATile), 16, 1024);
    if (lead && tc::elect_one()) {
      auto wait1 = [&](uint64_t* b_, uint32_t par) { return tc::mbar_wait(b_, par, abort_flag, &g_status_lmh); };
      int q = 0, nt = 0;  // stages consumed, tiles accumulated
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (!(ok = wait1(item_full + (k & 1), (k >> 1) & 1))) break;
        const int it = item_ring[k & 1];
        tc::mbar_arrive(item_empty + (k & 1));
        if (it < 0) break;
        const LmhItem I = decode(p, it);
        const int vt1 = min(p.n_vt, (I.vc + 1) * kVt);
        for (int vt = I.vc * kVt; ok && vt < vt1; ++vt, ++nt) {
          const int ab = nt & 1;
          if (nt >= 2 && !(ok = wait1(acc_free + ab, ((nt >> 1) - 1) & 1))) break;
          for (int kc = 0; kc < n_k; ++kc, ++q) {
            const int s = q % kStages;
            if (!(ok = wait1(full + s, (q / kStages) & 1))) break;
            tc::tc_fence_after();
            const uint32_t so = (s * kStage) >> 4;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              tc::mma2_ss(tmem + 256 * ab, dA + so + ((kk * 32) >> 4), dB + so + ((kk * 32) >> 4), idesc,
                          (kc > 0 || kk > 0) ? 1u : 0u);
            tc::mma2_commit_both(empty + s);
            if (kc + 1 == n_k) tc::mma2_commit_both(acc_full + ab);
          }
        }
      }
      if (*abort_flag) {  // let issued MMAs finish before TMEM is released
        volatile int never = 0;
        tc::mma2_commit_both(drain);
        tc::mbar_wait(drain, 0, &never, &g_status_lmh, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue warpgroups
    const int w = warp >> 2;          // vocab columns [64w, 64w+64) of each tile
    const int r = threadIdx.x & 127;  // row of the tile = TMEM lane
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    int nt = 0, ni = 0;  // tiles and items with work processed
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!wait_ring(item_full + (k & 1), (k >> 1) & 1)) break;
      const int it = item_ring[k & 1];
      warp_arrive_lead(item_empty + (k & 1));
      if (it < 0) break;
      const LmhItem I = decode(p, it);
      const int64_t row = int64_t(I.rt) * 2 * kBM + kBM * int(crank) + r;
      const bool real = row < p.rows;
      // children of this row: their tokens are its labels
      int b = 0, pos = 0, c0 = 0, c1 = 0, lmin = 0x7fffffff, lmax = -1;
      if (real) {
        row_to_pos(p, row, b, pos);
        c0 = p.child_off[int64_t(b) * (p.t_pad + 1) + pos];
        c1 = p.child_off[int64_t(b) * (p.t_pad + 1) + pos + 1];
        if (!dbg_ok(c0 >= 0 && c0 <= c1 && c1 <= p.t_pad, &g_status_lmh)) c1 = c0;
        for (int c = c0; c < c1; ++c) {
          const int cp = p.child_pos[int64_t(b) * p.t_pad + c];
          if (!dbg_ok(cp > pos && cp < p.t_pad, &g_status_lmh)) {
            c1 = c;  // labels from here on are not read
            break;
          }
          const int tok = p.tokens[int64_t(b) * p.t_pad + cp];
          lmin = min(lmin, tok);
          lmax = max(lmax, tok);
        }
      }
      Stats st{-INFINITY, 0.f, 0.f};
      const int vt1 = min(p.n_vt, (I.vc + 1) * kVt);
      for (int vt = I.vc * kVt; vt < vt1; ++vt, ++nt) {
        const int ab = nt & 1;
        if (!wait_u(acc_full + ab, (nt >> 1) & 1)) { ok = false; break; }
        tc::tc_fence_after();
        const int v0 = vt * kBN + 64 * w;  // vocab index of this thread's first column
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t x[32];
          tc::tmem_ld32(tmem + lane_base + 256 * ab + 64 * w + 32 * h, x);
          tc::tmem_ld_wait();
          if (h == 1) {
            tc::tc_fence_before();
            warp_arrive_lead(acc_free + ab);  // both halves are in registers
          }
          const int vb = v0 + 32 * h;
          float mx = -INFINITY;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (vb + c >= p.vocab) x[c] = __float_as_uint(-INFINITY);
            mx = fmaxf(mx, __uint_as_float(x[c]));
          }
          if (mx > st.m) {
            const float cf = tc::ex2((st.m - mx) * kLog2e);
            st.s *= cf;
            st.t *= cf;
            st.m = mx;
          }
          if (st.m > -INFINITY) {
            const float mb = st.m * kLog2e;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float xv = __uint_as_float(x[c]);
              const float e = tc::ex2(fmaf(xv, kLog2e, -mb));
              st.s += e;
              st.t = (vb + c < p.vocab) ? fmaf(e, xv, st.t) : st.t;
            }
          }
          if (real && lmax >= vb && lmin < vb + 32) {  // a label may fall in these 32 columns
            for (int c = c0; c < c1; ++c) {
              const int cp = p.child_pos[int64_t(b) * p.t_pad + c];
              const int col = p.tokens[int64_t(b) * p.t_pad + cp] - vb;
              if (col >= 0 && col < 32) {
                uint32_t v = x[0];
#pragma unroll
                for (int j = 1; j < 32; ++j) v = (col == j) ? x[j] : v;
                p.pair_logit[int64_t(b) * p.t_pad + cp] = __uint_as_float(v);
              }
            }
          }
        }
      }
      if (!ok) break;
      // Merge the four warpgroups' statistics of each row into one partial,
      // through a buffer that alternates by item.
      float4* mb = sMerge + (ni & 1) * 3 * kBM;
      if (w > 0) {
        if (ni >= 2 && !wait_u(merge_free + (ni & 1), ((ni >> 1) - 1) & 1)) { ok = false; break; }
        mb[(w - 1) * kBM + r] = make_float4(st.m, st.s, st.t, 0.f);
        tc::mbar_arrive(merge_full + (ni & 1));
      } else {
        if (!wait_u(merge_full + (ni & 1), (ni >> 1) & 1)) { ok = false; break; }
        if (real) {
          Stats a = st;
          for (int u = 0; u < 3; ++u) {
            const float4 o = mb[u * kBM + r];
            stats_merge(a, Stats{o.x, o.y, o.z});
          }
          p.part[row * p.n_vc + I.vc] = make_float4(a.m, a.s, a.t, 0.f);
        }
        tc::mbar_arrive(merge_free + (ni & 1));
      }
      ++ni;
    }
  }

  tc::tc_fence_before();
  tc::cluster_sync();  // the pair's MMAs into either CTA's TMEM are done before it is freed
  tc::tc_fence_after();
  if (warp == kWMma) tc::tmem_dealloc2(tmem, 512);
}

// One thread per tree position (b, pos): merges its row's partials; writes its
// entropy, the log-probs of its children, and 0 where nothing is defined.
__global__ void __launch_bounds__(256) lmh_combine_kernel(const LmhParams p, const int32_t* __restrict__ parent,
                                                         float* __restrict__ pos_logp,
                                                         float* __restrict__ pos_entropy) {
  const int64_t at = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (at >= int64_t(p.n_trees) * p.t_pad) return;
  const int b = int(at / p.t_pad), pos = int(at % p.t_pad);
  if (pos >= p.n_tokens[b]) {
    pos_logp[at] = 0.f;
    pos_entropy[at] = 0.f;
    return;
  }
  const int64_t row = p.tok_base[b] + pos;
  if (!dbg_ok(row >= 0 && row < p.rows, &g_status_lmh)) return;
  Stats a{-INFINITY, 0.f, 0.f};
  for (int vc = 0; vc < p.n_vc; ++vc) {
    const float4 o = p.part[row * p.n_vc + vc];
    stats_merge(a, Stats{o.x, o.y, o.z});
  }
  const float lse = a.m + __log2f(a.s) * kLn2;
  pos_entropy[at] = lse - a.t / a.s;
  if (parent[at] < 0) pos_logp[at] = 0.f;  // no parent row: no label
  const int c0 = p.child_off[int64_t(b) * (p.t_pad + 1) + pos];
  const int c1 = p.child_off[int64_t(b) * (p.t_pad + 1) + pos + 1];
  if (!dbg_ok(c0 >= 0 && c0 <= c1 && c1 <= p.t_pad, &g_status_lmh)) return;
  for (int c = c0; c < c1; ++c) {
    const int cp = p.child_pos[int64_t(b) * p.t_pad + c];
    if (!dbg_ok(cp > pos && cp < p.n_tokens[b], &g_status_lmh)) continue;
    const int tok = p.tokens[int64_t(b) * p.t_pad + cp];
    pos_logp[int64_t(b) * p.t_pad + cp] =
        (tok >= 0 && tok < p.vocab) ? p.pair_logit[int64_t(b) * p.t_pad + cp] - lse : __int_as_float(0x7fc00000);
  }
}

int num_sms_lmh() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 148;
  }
  return sms;
}

inline uint64_t al256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

}  // namespace

TPA_DEFINE_STATUS_READER(tpa_internal_status_lmh, g_status_lmh)

extern "C" uint64_t tpa_lm_head_workspace_bytes(int64_t rows, int32_t vocab, int32_t n_trees, int32_t t_pad) {
  if (rows < 1 || vocab < 1 || n_trees < 1 || t_pad < 1) return 0;
  const uint64_t n_vt = (uint64_t(vocab) + kBN - 1) / kBN;
  const uint64_t n_vc = (n_vt + kVt - 1) / kVt;
  return 256 + al256(uint64_t(rows) * n_vc * 16) + al256(uint64_t(n_trees) * uint64_t(t_pad) * 4);
}

extern "C" int tpa_lm_head_logprobs_entropy(const tpa_tree_view* tree, const void* hidden, const void* weight,
                                            int32_t hidden_size, int32_t vocab, void* workspace,
                                            uint64_t workspace_bytes, float* pos_logp, float* pos_entropy,
                                            float* seq_logp, float* seq_entropy, void* stream) {
  TPA_NVTX_RANGE("tpa_lm_head_logprobs_entropy");
  if (!tree || !hidden || !weight || !workspace || !pos_logp || !pos_entropy || !seq_logp || !seq_entropy)
    return TPA_ERR_INVALID_ARG;
  if (tree->n_trees < 1 || tree->t_pad < 1 || tree->n_seqs < 1 || tree->total_tree_tokens < 1)
    return TPA_ERR_INVALID_ARG;
  if (hidden_size < kBK || hidden_size % kBK != 0 || hidden_size > 65536 || vocab < 1) return TPA_ERR_INVALID_ARG;
  if (tree->max_token < 0 || tree->max_token >= vocab) return TPA_ERR_INVALID_ARG;  // a label past the vocabulary
  if ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(weight)) & 15) return TPA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return TPA_ERR_INVALID_ARG;
  const int64_t rows = tree->total_tree_tokens;
  if (workspace_bytes < tpa_lm_head_workspace_bytes(rows, vocab, tree->n_trees, tree->t_pad))
    return TPA_ERR_BUFFER_TOO_SMALL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  LmhParams p;
  p.n_tokens = tree->n_tokens;
  p.tok_base = tree->tok_base;
  p.tokens = tree->tokens;
  p.child_off = tree->child_off;
  p.child_pos = tree->child_pos;
  p.rows = rows;
  p.n_trees = tree->n_trees;
  p.t_pad = tree->t_pad;
  p.vocab = vocab;
  p.hidden = hidden_size;
  p.n_rt = int((rows + 2 * kBM - 1) / (2 * kBM));  // 256-row tiles of a CTA pair
  p.n_vt = (vocab + kBN - 1) / kBN;
  p.n_vc = (p.n_vt + kVt - 1) / kVt;
  // rows of a group: their hidden tiles (256 x H bf16 each) take about 48 MB of L2
  const int64_t per_tile = int64_t(2 * kBM) * hidden_size * 2;
  p.group = int(std::max<int64_t>(1, std::min<int64_t>(p.n_rt, (int64_t(48) << 20) / per_tile)));
  p.n_items = p.n_rt * p.n_vc;
  p.ctr = reinterpret_cast<uint32_t*>(ws);
  p.part = reinterpret_cast<float4*>(ws + 256);
  p.pair_logit = reinterpret_cast<float*>(ws + 256 + al256(uint64_t(rows) * p.n_vc * 16));
  CUtensorMap tm_h, tm_w;
  if (!tmap::make_rows_heads_d(&tm_h, hidden, uint64_t(rows), 1, uint64_t(hidden_size), kBM) ||
      !tmap::make_rows_heads_d(&tm_w, weight, uint64_t(vocab), 1, uint64_t(hidden_size), kBN / 2))
    return TPA_ERR_CUDA;
  TPA_CUDA_TRY(cudaMemsetAsync(ws, 0, 16, st));
  TPA_CUDA_TRY(cudaFuncSetAttribute(lmh_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes));
  const int pairs = std::max(1, num_sms_lmh() / 2);
  lmh_kernel<<<2 * (p.n_items < pairs ? p.n_items : pairs), kThreads, kSmemBytes, st>>>(tm_h, tm_w, p);
  TPA_CUDA_TRY(cudaGetLastError());
  const int64_t n_pos = int64_t(tree->n_trees) * tree->t_pad;
  lmh_combine_kernel<<<int((n_pos + 255) / 256), 256, 0, st>>>(p, tree->parent, pos_logp, pos_entropy);
  TPA_CUDA_TRY(cudaGetLastError());
  return tpa_internal_seq_gather(tree, pos_logp, pos_entropy, seq_logp, seq_entropy, stream);
}
