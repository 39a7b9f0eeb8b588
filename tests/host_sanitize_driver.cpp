// Host-side exercise of libtpa's packer, extraction and balancing code,
// compiled together with pack.cpp and balance.cpp under AddressSanitizer and
// UndefinedBehaviorSanitizer by tests/test_host_sanitizers.py.  It runs the
// worked example of the tree-training page (§树构建过程: [A,B,C,D],
// [A,B,E,F], [A,G,H] give 8 tree tokens of 11), seeded random sequence sets
// over tiny vocabularies (heavy sharing, many trees, sequences ending inside
// nodes), padded batches, every argument error path, and FFD / KK balancing
// with the packing metrics.  It checks a few invariants that hold for any
// input and exits non-zero on the first violation; the sanitizers abort on
// any out-of-bounds access, leak, overflow or misaligned access.
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "tpa.h"

namespace {

uint64_t rng_state = 0x9E3779B97F4A7C15ull;
uint64_t next_u64() {  // splitmix64
  uint64_t z = (rng_state += 0x9E3779B97F4A7C15ull);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}
int uniform(int lo, int hi) { return lo + int(next_u64() % uint64_t(hi - lo + 1)); }

#define CHECK(cond)                                                       \
  do {                                                                    \
    if (!(cond)) {                                                        \
      std::fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      std::exit(1);                                                       \
    }                                                                     \
  } while (0)

// Every view array of every tree is read once, and the layout invariants that
// hold for any packing are checked: preorder parents precede children, each
// position's subtree end covers it, pad positions are marked.
void check_tree(const tpa_tree* t, int64_t total_tokens) {
  tpa_tree_info info;
  CHECK(tpa_tree_get_info(t, &info) == TPA_OK);
  CHECK(info.total_seq_tokens == total_tokens);
  CHECK(info.total_tree_tokens <= total_tokens && info.total_tree_tokens >= 1);
  tpa_tree_view v;
  CHECK(tpa_tree_make_view(t, tpa_tree_host_blob(t), &v) == TPA_OK);
  const int64_t T = info.t_pad;
  int64_t pairs = 0;
  for (int b = 0; b < info.n_trees; ++b) {
    const int n = v.n_tokens[b];
    CHECK(n >= 1 && n <= T);
    CHECK(v.tok_base[b + 1] - v.tok_base[b] == n);
    for (int64_t p = 0; p < T; ++p) {
      const int64_t at = b * T + p;
      if (p < n) {
        CHECK(v.tokens[at] >= 0 && v.tokens[at] <= info.max_token);
        CHECK(v.parent[at] < p);
        CHECK(v.subtree_end[at] >= p && v.subtree_end[at] < n);
        CHECK(v.depth[at] == (v.parent[at] < 0 ? 0 : v.depth[b * T + v.parent[at]] + 1));
        CHECK(v.node_id[at] >= 0 && v.node_id[at] < v.n_nodes[b]);
        pairs += v.depth[at] + 1;
        const int32_t* co = v.child_off + b * (T + 1);
        for (int c = co[p]; c < co[p + 1]; ++c) CHECK(v.parent[b * T + v.child_pos[b * T + c]] == p);
      } else {
        CHECK(v.tokens[at] == -1 && v.subtree_end[at] == -1 && v.parent[at] == -1 && v.node_id[at] == -1);
      }
    }
    for (int k = 0; k < v.n_nodes[b]; ++k) {
      const int32_t* ni = v.node_info + (int64_t(b) * info.max_nodes + k) * 4;
      CHECK(ni[0] <= ni[1] && ni[1] <= ni[3] && ni[3] < n);
    }
  }
  CHECK(pairs == info.ancestor_pairs && v.ancestor_pairs == pairs);
  for (int s = 0; s < info.n_seqs; ++s) {
    CHECK(v.seq_tree[s] >= 0 && v.seq_tree[s] < info.n_trees);
    for (int64_t i = v.seq_off[s]; i < v.seq_off[s + 1]; ++i) {
      CHECK(v.seq_pos[i] >= 0 && v.seq_pos[i] < v.n_tokens[v.seq_tree[s]]);
      if (i > v.seq_off[s]) CHECK(v.parent[int64_t(v.seq_tree[s]) * T + v.seq_pos[i]] == v.seq_pos[i - 1]);
    }
  }
}

void worked_example() {
  // A=1 B=2 C=3 D=4 E=5 F=6 G=7 H=8
  const int32_t tokens[] = {1, 2, 3, 4, 1, 2, 5, 6, 1, 7, 8};
  const int64_t offs[] = {0, 4, 8, 11};
  tpa_tree* t = nullptr;
  CHECK(tpa_tree_pack(tokens, offs, 3, 128, &t) == TPA_OK && t);
  tpa_tree_info info;
  CHECK(tpa_tree_get_info(t, &info) == TPA_OK);
  CHECK(info.n_trees == 1 && info.total_tree_tokens == 8 && info.total_seq_tokens == 11);
  check_tree(t, 11);
  tpa_tree_free(t);
}

void random_sets() {
  for (int round = 0; round < 300; ++round) {
    const int n = uniform(1, 40), vocab = uniform(1, 5), max_len = uniform(1, 300);
    const int mb = 128 * uniform(1, 4);
    std::vector<int32_t> toks;
    std::vector<int64_t> offs{0};
    for (int s = 0; s < n; ++s) {
      const int L = uniform(1, max_len < mb ? max_len : mb);
      for (int i = 0; i < L; ++i) toks.push_back(uniform(0, vocab - 1) * (round % 7 == 0 ? 100003 : 1));
      offs.push_back(int64_t(toks.size()));
    }
    tpa_tree* t = nullptr;
    CHECK(tpa_tree_pack(toks.data(), offs.data(), n, mb, &t) == TPA_OK);
    check_tree(t, int64_t(toks.size()));
    tpa_tree_free(t);

    // the same sequences as a left/right-padded batch
    int row_len = 0;
    for (int s = 0; s < n; ++s) row_len = int(offs[s + 1] - offs[s]) > row_len ? int(offs[s + 1] - offs[s]) : row_len;
    row_len += 3;
    std::vector<int32_t> ids(size_t(n) * row_len, 77);
    std::vector<uint8_t> am(size_t(n) * row_len, 0);
    for (int s = 0; s < n; ++s) {
      const int L = int(offs[s + 1] - offs[s]);
      const int lead = (s % 2) ? row_len - L : 0;
      for (int i = 0; i < L; ++i) {
        ids[size_t(s) * row_len + lead + i] = toks[offs[s] + i];
        am[size_t(s) * row_len + lead + i] = 1;
      }
    }
    std::vector<int32_t> out_tok(size_t(n) * row_len);
    std::vector<int64_t> out_off(n + 1);
    CHECK(tpa_extract_sequences(ids.data(), am.data(), n, row_len, out_tok.data(), out_off.data()) == TPA_OK);
    CHECK(out_off[n] == offs[n]);
    for (int64_t i = 0; i < offs[n]; ++i) CHECK(out_tok[i] == toks[i]);
    tpa_tree* t2 = nullptr;
    CHECK(tpa_tree_pack_padded(ids.data(), am.data(), n, row_len, mb, &t2) == TPA_OK);
    check_tree(t2, int64_t(toks.size()));
    tpa_tree_free(t2);
  }
}

void error_paths() {
  const int32_t toks[] = {1, 2, 3};
  const int64_t offs[] = {0, 3};
  const int64_t empty_offs[] = {0, 0};
  const int64_t bad_offs[] = {1, 3};
  tpa_tree* t = reinterpret_cast<tpa_tree*>(0x1);
  CHECK(tpa_tree_pack(toks, offs, 1, 100, &t) == TPA_ERR_INVALID_ARG && t == nullptr);
  CHECK(tpa_tree_pack(toks, offs, 0, 128, &t) == TPA_ERR_INVALID_ARG);
  CHECK(tpa_tree_pack(nullptr, offs, 1, 128, &t) == TPA_ERR_INVALID_ARG);
  CHECK(tpa_tree_pack(toks, empty_offs, 1, 128, &t) == TPA_ERR_EMPTY_SEQUENCE);
  CHECK(tpa_tree_pack(toks, bad_offs, 1, 128, &t) == TPA_ERR_INVALID_ARG);
  CHECK(tpa_tree_pack(toks, offs, 1, 128, nullptr) == TPA_ERR_INVALID_ARG);
  std::vector<int32_t> long_seq(200, 4);
  const int64_t long_offs[] = {0, 200};
  CHECK(tpa_tree_pack(long_seq.data(), long_offs, 1, 128, &t) == TPA_ERR_SEQ_TOO_LONG);
  const int32_t neg[] = {1, -2, 3};
  CHECK(tpa_tree_pack(neg, offs, 1, 128, &t) == TPA_ERR_INVALID_ARG);
  tpa_tree_info info;
  CHECK(tpa_tree_get_info(nullptr, &info) == TPA_ERR_INVALID_ARG);
  tpa_tree_free(nullptr);
  const uint8_t none[3] = {0, 0, 0};
  CHECK(tpa_tree_pack_padded(toks, none, 1, 3, 128, &t) == TPA_ERR_EMPTY_SEQUENCE);
}

void balancing() {
  for (int round = 0; round < 300; ++round) {
    const int n = uniform(1, 64);
    std::vector<int64_t> w(n);
    int64_t mx = 0, total = 0;
    for (auto& x : w) {
      x = (next_u64() % 10 < 3) ? uniform(800, 2048) : uniform(50, 200);
      mx = x > mx ? x : mx;
      total += x;
    }
    const int64_t cap = (round % 2) ? mx + uniform(0, 3000) : total * 4;
    const int min_groups = uniform(1, n < 8 ? n : 8), div = uniform(1, 3);
    for (int algo = 0; algo < 2; ++algo) {
      std::vector<int32_t> g(n, -1);
      int32_t ng = 0, used = -1;
      const int rc = tpa_balance(w.data(), n, cap, min_groups, div, algo, g.data(), &ng, &used);
      if (rc != TPA_OK) {
        CHECK(rc == TPA_ERR_INVALID_ARG);  // more groups required than items
        continue;
      }
      CHECK(ng >= min_groups && ng % div == 0 && (used == 0 || used == 1));
      std::vector<int64_t> load(ng, 0);
      for (int i = 0; i < n; ++i) {
        CHECK(g[i] >= 0 && g[i] < ng);
        load[g[i]] += w[i];
      }
      for (int64_t l : load) CHECK(l <= cap);
      tpa_packing_metrics_t m;
      CHECK(tpa_packing_metrics(w.data(), n, g.data(), ng, cap, &m) == TPA_OK);
      CHECK(m.total == total && m.spread == m.max_load - m.min_load && m.n_groups == ng);
    }
  }
  int32_t g[1], ng = 0;
  const int64_t heavy[] = {10};
  CHECK(tpa_balance(heavy, 1, 5, 1, 1, 0, g, &ng, nullptr) == TPA_ERR_SEQ_TOO_LONG);
  CHECK(tpa_balance(heavy, 1, 50, 1, 1, 9, g, &ng, nullptr) == TPA_ERR_INVALID_ARG);
  CHECK(tpa_balance(nullptr, 1, 50, 1, 1, 0, g, &ng, nullptr) == TPA_ERR_INVALID_ARG);
}

}  // namespace

int main() {
  worked_example();
  random_sets();
  error_paths();
  balancing();
  std::printf("host sanitize driver: ok\n");
  return 0;
}
