// Host trie packer of libtpa (tpa_tree_pack and the tree handle API).
//
// Tree training page (AReaL "树训练"), §树构建过程: sequences are inserted
// greedily into prefix tries with a first-fit-decreasing policy (step 2), and
// linear chains are merged into compressed nodes (step 3); §数据结构 TrieNode:
// nodes hold inclusive [start_idx, end_idx] ranges of a preorder flattening,
// children keyed by branching token; §配置: a tree holds at most
// max_tokens_per_mb tokens, a multiple of 128.
//
// Data structures: one vertex-array trie per tree with an open-addressing
// (vertex, token) -> child table and intrusive sibling lists that keep the
// children in insertion order.  The whole result is written into one
// 256-byte-aligned int32/int64 blob whose sections the view functions slice.
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <numeric>
#include <vector>

#include "tpa.h"
#include "internal.h"

namespace {

constexpr int32_t kMaxTPad = 131072;  // n_blk <= 1024 (limit of the CSR builder)

// Open-addressing map from (parent vertex, token) to child vertex.
class ChildTable {
 public:
  ChildTable() { rehash(1024); }

  int32_t find(int32_t v, int32_t tok) const {
    const uint64_t key = pack(v, tok);
    for (uint64_t h = mix(key) & mask_;; h = (h + 1) & mask_) {
      if (keys_[h] == kEmpty) return -1;
      if (keys_[h] == key) return vals_[h];
    }
  }

  void insert(int32_t v, int32_t tok, int32_t child) {
    if ((used_ + 1) * 2 > keys_.size()) rehash(keys_.size() * 2);
    place(pack(v, tok), child);
    ++used_;
  }

 private:
  static constexpr uint64_t kEmpty = ~0ull;
  static uint64_t pack(int32_t v, int32_t tok) {
    return (uint64_t(uint32_t(v)) << 32) | uint32_t(tok);
  }
  static uint64_t mix(uint64_t x) {  // splitmix64 finaliser
    x ^= x >> 30; x *= 0xbf58476d1ce4e5b9ull;
    x ^= x >> 27; x *= 0x94d049bb133111ebull;
    return x ^ (x >> 31);
  }
  void place(uint64_t key, int32_t val) {
    uint64_t h = mix(key) & mask_;
    while (keys_[h] != kEmpty) h = (h + 1) & mask_;
    keys_[h] = key;
    vals_[h] = val;
  }
  void rehash(size_t cap) {
    std::vector<uint64_t> ok;
    std::vector<int32_t> ov;
    ok.swap(keys_);
    ov.swap(vals_);
    keys_.assign(cap, kEmpty);
    vals_.assign(cap, -1);
    mask_ = cap - 1;
    for (size_t i = 0; i < ok.size(); ++i)
      if (ok[i] != kEmpty) place(ok[i], ov[i]);
  }
  std::vector<uint64_t> keys_;
  std::vector<int32_t> vals_;
  uint64_t mask_ = 0;
  size_t used_ = 0;
};

// Uncompressed token trie; vertex 0 is the root.  A vertex's first child is
// found through `first`; only its later children (the branch points) go into
// the hash table, so walking or extending a chain does no hashing.
struct Trie {
  std::vector<int32_t> tok{-1}, par{-1}, first{-1}, last{-1}, next{-1}, nchild{0};
  ChildTable table;
  std::vector<int32_t> members;  // input sequence ids, in insertion order

  int32_t n_tokens() const { return int32_t(tok.size()) - 1; }

  int32_t child(int32_t v, int32_t t) const {
    const int32_t c = first[v];
    if (c < 0) return -1;
    if (tok[c] == t) return c;
    return nchild[v] > 1 ? table.find(v, t) : -1;
  }

  // Whether the first `need` tokens of s are a path from the root: the
  // sequence then adds at most len - need new tokens.
  bool shares_at_least(const int32_t* s, int64_t need) const {
    int32_t v = 0;
    for (int64_t n = 0; n < need; ++n) {
      v = child(v, s[n]);
      if (v < 0) return false;
    }
    return true;
  }

  void insert(const int32_t* s, int64_t len, int32_t* vertex_out) {
    int32_t v = 0;
    for (int64_t t = 0; t < len; ++t) {
      int32_t c = child(v, s[t]);
      if (c < 0) {
        c = int32_t(tok.size());
        tok.push_back(s[t]);
        par.push_back(v);
        first.push_back(-1);
        last.push_back(-1);
        next.push_back(-1);
        nchild.push_back(0);
        if (last[v] < 0) {
          first[v] = c;
        } else {
          next[last[v]] = c;
          table.insert(v, s[t], c);  // a second or later child
        }
        last[v] = c;
        ++nchild[v];
      }
      vertex_out[t] = c;
      v = c;
    }
  }
};

// Blob sections, in order.
enum Section {
  kTokens, kSubtreeEnd, kParent, kDepth, kNodeId, kChildOff, kChildPos, kNTokens,
  kTokBase, kNodeInfo, kNNodes, kSeqTree, kSeqOff, kSeqPos, kNumSections
};

inline uint64_t align256(uint64_t x) { return (x + 255) & ~uint64_t(255); }

}  // namespace

struct tpa_tree {
  tpa_tree_info info{};
  uint64_t off[kNumSections + 1]{};
  uint8_t* blob = nullptr;
  ~tpa_tree() { std::free(blob); }
};

namespace {

void compute_layout(tpa_tree* t) {
  const uint64_t B = uint64_t(t->info.n_trees), T = uint64_t(t->info.t_pad);
  const uint64_t S = uint64_t(t->info.n_seqs), N = uint64_t(t->info.total_seq_tokens);
  const uint64_t M = uint64_t(t->info.max_nodes);
  const uint64_t bytes[kNumSections] = {
      4 * B * T, 4 * B * T, 4 * B * T, 4 * B * T, 4 * B * T, 4 * B * (T + 1), 4 * B * T,
      4 * B, 8 * (B + 1), 16 * B * M, 4 * B, 4 * S, 8 * (S + 1), 4 * N};
  uint64_t o = 0;
  for (int i = 0; i < kNumSections; ++i) {
    t->off[i] = o;
    o = align256(o + bytes[i]);
  }
  t->off[kNumSections] = o;
  t->info.blob_bytes = o;
}

template <typename T>
T* sect(tpa_tree* t, int s) { return reinterpret_cast<T*>(t->blob + t->off[s]); }

int pack_impl(const int32_t* tokens, const int64_t* offs, int32_t n_seqs, int32_t mb,
              tpa_tree** out) {
  if (!out) return TPA_ERR_INVALID_ARG;
  *out = nullptr;
  if (!tokens || !offs || n_seqs < 1 || mb <= 0 || mb % TPA_BLOCK_SIZE != 0 || mb > kMaxTPad)
    return TPA_ERR_INVALID_ARG;
  if (offs[0] != 0) return TPA_ERR_INVALID_ARG;
  for (int32_t s = 0; s < n_seqs; ++s) {
    const int64_t len = offs[s + 1] - offs[s];
    if (len < 0) return TPA_ERR_INVALID_ARG;
    if (len == 0) return TPA_ERR_EMPTY_SEQUENCE;
    if (len > mb) return TPA_ERR_SEQ_TOO_LONG;
  }
  const int64_t total = offs[n_seqs];
  int32_t max_token = 0;
  for (int64_t i = 0; i < total; ++i) {
    if (tokens[i] < 0) return TPA_ERR_INVALID_ARG;
    max_token = std::max(max_token, tokens[i]);
  }

  // Longest first; equal lengths keep input order.
  std::vector<int32_t> order(n_seqs);
  std::iota(order.begin(), order.end(), 0);
  std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
    return (offs[a + 1] - offs[a]) > (offs[b + 1] - offs[b]);
  });

  std::vector<Trie> tries;
  std::vector<int32_t> seq_tree(n_seqs);
  std::vector<int32_t> seq_vertex(static_cast<size_t>(total));  // trie vertex of every input token
  for (int32_t s : order) {
    const int32_t* seq = tokens + offs[s];
    const int64_t len = offs[s + 1] - offs[s];
    // First fit: the first tree whose token count plus the sequence's new
    // tokens (those past its shared prefix) stays within mb.  A tree with room
    // for the whole sequence takes it without a walk; otherwise the walk stops
    // once the prefix is long enough or the trie ends.
    size_t b = 0;
    for (; b < tries.size(); ++b) {
      const int64_t room = int64_t(mb) - tries[b].n_tokens();
      if (len <= room || tries[b].shares_at_least(seq, len - room)) break;
    }
    if (b == tries.size()) tries.emplace_back();
    tries[b].insert(seq, len, seq_vertex.data() + offs[s]);
    tries[b].members.push_back(s);
    seq_tree[s] = int32_t(b);
  }

  const int32_t B = int32_t(tries.size());
  const int64_t T = mb;
  // Per tree: preorder positions, then the flat arrays.
  std::vector<std::vector<int32_t>> pos_of(B);
  std::vector<std::vector<int32_t>> ordv(B);
  int32_t max_nodes = 0;
  for (int32_t b = 0; b < B; ++b) {
    const Trie& tr = tries[b];
    const int32_t nv = int32_t(tr.tok.size());
    auto& pos = pos_of[b];
    auto& ord = ordv[b];
    pos.assign(nv, -1);
    ord.reserve(nv - 1);
    std::vector<int32_t> stack;
    // push children of v so that the first-inserted child is popped first
    auto push_children = [&](int32_t v) {
      const size_t base = stack.size();
      for (int32_t c = tr.first[v]; c >= 0; c = tr.next[c]) stack.push_back(c);
      std::reverse(stack.begin() + base, stack.end());
    };
    push_children(0);
    while (!stack.empty()) {
      const int32_t v = stack.back();
      stack.pop_back();
      pos[v] = int32_t(ord.size());
      ord.push_back(v);
      push_children(v);
    }
    int32_t nn = 0;
    for (int32_t p = 0; p < int32_t(ord.size()); ++p) {
      const int32_t pv = tr.par[ord[p]];
      if (pv == 0 || tr.nchild[pv] != 1) ++nn;
    }
    max_nodes = std::max(max_nodes, nn);
  }

  tpa_tree* t = new tpa_tree();
  t->info.n_trees = B;
  t->info.t_pad = mb;
  t->info.n_seqs = n_seqs;
  t->info.max_nodes = max_nodes;
  t->info.total_seq_tokens = total;
  t->info.max_token = max_token;
  compute_layout(t);
  t->blob = static_cast<uint8_t*>(std::aligned_alloc(256, t->info.blob_bytes));
  if (!t->blob) { delete t; return TPA_ERR_NO_MEMORY; }
  std::memset(t->blob, 0, t->info.blob_bytes);

  int32_t* tok_a = sect<int32_t>(t, kTokens);
  int32_t* end_a = sect<int32_t>(t, kSubtreeEnd);
  int32_t* par_a = sect<int32_t>(t, kParent);
  int32_t* dep_a = sect<int32_t>(t, kDepth);
  int32_t* nid_a = sect<int32_t>(t, kNodeId);
  int32_t* coff_a = sect<int32_t>(t, kChildOff);
  int32_t* cpos_a = sect<int32_t>(t, kChildPos);
  int32_t* ntok_a = sect<int32_t>(t, kNTokens);
  int64_t* base_a = sect<int64_t>(t, kTokBase);
  int32_t* ninfo_a = sect<int32_t>(t, kNodeInfo);
  int32_t* nnod_a = sect<int32_t>(t, kNNodes);
  std::fill(tok_a, tok_a + B * T, -1);
  std::fill(end_a, end_a + B * T, -1);
  std::fill(par_a, par_a + B * T, -1);
  std::fill(nid_a, nid_a + B * T, -1);
  std::fill(cpos_a, cpos_a + B * T, -1);
  std::fill(ninfo_a, ninfo_a + int64_t(B) * max_nodes * 4, -1);

  int64_t tree_tokens = 0, nodes_total = 0, pairs = 0;
  base_a[0] = 0;
  for (int32_t b = 0; b < B; ++b) {
    const Trie& tr = tries[b];
    const auto& pos = pos_of[b];
    const auto& ord = ordv[b];
    const int32_t n = int32_t(ord.size());
    int32_t* tk = tok_a + b * T;
    int32_t* en = end_a + b * T;
    int32_t* pa = par_a + b * T;
    int32_t* de = dep_a + b * T;
    int32_t* ni = nid_a + b * T;
    int32_t* co = coff_a + b * (T + 1);
    int32_t* cp = cpos_a + b * T;
    for (int32_t p = 0; p < n; ++p) {
      const int32_t v = ord[p];
      tk[p] = tr.tok[v];
      pa[p] = tr.par[v] == 0 ? -1 : pos[tr.par[v]];
      de[p] = pa[p] < 0 ? 0 : de[pa[p]] + 1;
      pairs += de[p] + 1;
    }
    // last position of each token's subtree (children follow parents)
    std::vector<int32_t> last(n);
    for (int32_t p = 0; p < n; ++p) last[p] = p;
    for (int32_t p = n - 1; p >= 0; --p)
      if (pa[p] >= 0) last[pa[p]] = std::max(last[pa[p]], last[p]);
    // compressed nodes
    int32_t* info = ninfo_a + int64_t(b) * max_nodes * 4;
    int32_t nn = 0;
    for (int32_t p = 0; p < n; ++p) {
      const int32_t pv = tr.par[ord[p]];
      if (pv != 0 && tr.nchild[pv] == 1) continue;
      int32_t q = p;
      while (tr.nchild[ord[q]] == 1) ++q;  // the single child is the next position
      for (int32_t r = p; r <= q; ++r) {
        ni[r] = nn;
        en[r] = last[p];
      }
      info[4 * nn + 0] = p;
      info[4 * nn + 1] = q;
      info[4 * nn + 2] = pa[p] < 0 ? -1 : ni[pa[p]];
      info[4 * nn + 3] = last[p];
      ++nn;
    }
    // children CSR, ascending child position
    std::vector<int32_t> cnt(n + 1, 0);
    for (int32_t c = 0; c < n; ++c)
      if (pa[c] >= 0) ++cnt[pa[c] + 1];
    co[0] = 0;
    for (int32_t p = 0; p < n; ++p) co[p + 1] = co[p] + cnt[p + 1];
    for (int64_t p = n; p < T; ++p) co[p + 1] = co[n];
    std::vector<int32_t> fill(co, co + n);
    for (int32_t c = 0; c < n; ++c)
      if (pa[c] >= 0) cp[fill[pa[c]]++] = c;
    ntok_a[b] = n;
    nnod_a[b] = nn;
    base_a[b + 1] = base_a[b] + n;
    tree_tokens += n;
    nodes_total += nn;
  }
  int32_t* st_a = sect<int32_t>(t, kSeqTree);
  int64_t* so_a = sect<int64_t>(t, kSeqOff);
  int32_t* sp_a = sect<int32_t>(t, kSeqPos);
  for (int32_t s = 0; s < n_seqs; ++s) {
    st_a[s] = seq_tree[s];
    const auto& pos = pos_of[seq_tree[s]];
    for (int64_t i = offs[s]; i < offs[s + 1]; ++i) sp_a[i] = pos[seq_vertex[i]];
  }
  for (int32_t s = 0; s <= n_seqs; ++s) so_a[s] = offs[s];

  t->info.total_tree_tokens = tree_tokens;
  t->info.total_nodes = nodes_total;
  t->info.ancestor_pairs = pairs;
  t->info.tree_token_ratio = double(tree_tokens) / double(total);
  *out = t;
  return TPA_OK;
}

}  // namespace

extern "C" {

int tpa_tree_pack(const int32_t* tokens, const int64_t* seq_offsets, int32_t n_seqs,
                  int32_t max_tokens_per_mb, tpa_tree** out) {
  TPA_NVTX_RANGE("tpa_tree_pack");
  try {
    return pack_impl(tokens, seq_offsets, n_seqs, max_tokens_per_mb, out);
  } catch (const std::bad_alloc&) {
    return TPA_ERR_NO_MEMORY;
  } catch (...) {
    return TPA_ERR_INVALID_ARG;
  }
}

// Step 1 of §树构建过程 (提取序列): the real tokens of a padded row are its
// input_ids entries whose attention_mask entry is non-zero, in column order
// (left padding, right padding and interior gaps alike).
int tpa_extract_sequences(const int32_t* input_ids, const uint8_t* attention_mask, int32_t n_rows,
                          int32_t row_len, int32_t* tokens_out, int64_t* offsets_out) {
  if (!input_ids || !attention_mask || !tokens_out || !offsets_out || n_rows < 1 || row_len < 1)
    return TPA_ERR_INVALID_ARG;
  int64_t n = 0;
  offsets_out[0] = 0;
  for (int32_t r = 0; r < n_rows; ++r) {
    const int64_t base = int64_t(r) * row_len;
    for (int32_t c = 0; c < row_len; ++c)
      if (attention_mask[base + c] != 0) tokens_out[n++] = input_ids[base + c];
    offsets_out[r + 1] = n;
  }
  return TPA_OK;
}

int tpa_tree_pack_padded(const int32_t* input_ids, const uint8_t* attention_mask, int32_t n_rows,
                         int32_t row_len, int32_t max_tokens_per_mb, tpa_tree** out) {
  TPA_NVTX_RANGE("tpa_tree_pack_padded");
  if (out) *out = nullptr;
  if (!input_ids || !attention_mask || !out || n_rows < 1 || row_len < 1) return TPA_ERR_INVALID_ARG;
  try {
    std::vector<int32_t> tokens(size_t(n_rows) * size_t(row_len));
    std::vector<int64_t> offsets(size_t(n_rows) + 1);
    const int rc = tpa_extract_sequences(input_ids, attention_mask, n_rows, row_len, tokens.data(),
                                         offsets.data());
    if (rc != TPA_OK) return rc;
    return pack_impl(tokens.data(), offsets.data(), n_rows, max_tokens_per_mb, out);
  } catch (const std::bad_alloc&) {
    return TPA_ERR_NO_MEMORY;
  } catch (...) {
    return TPA_ERR_INVALID_ARG;
  }
}

int tpa_tree_get_info(const tpa_tree* tree, tpa_tree_info* info) {
  if (!tree || !info) return TPA_ERR_INVALID_ARG;
  *info = tree->info;
  return TPA_OK;
}

const void* tpa_tree_host_blob(const tpa_tree* tree) { return tree ? tree->blob : nullptr; }

int tpa_tree_make_view(const tpa_tree* tree, const void* base, tpa_tree_view* v) {
  if (!tree || !base || !v) return TPA_ERR_INVALID_ARG;
  const uint8_t* b = static_cast<const uint8_t*>(base);
  const uint64_t* o = tree->off;
  v->n_trees = tree->info.n_trees;
  v->t_pad = tree->info.t_pad;
  v->n_seqs = tree->info.n_seqs;
  v->max_nodes = tree->info.max_nodes;
  v->total_seq_tokens = tree->info.total_seq_tokens;
  v->total_tree_tokens = tree->info.total_tree_tokens;
  v->max_token = tree->info.max_token;
  v->reserved_ = 0;
  v->ancestor_pairs = tree->info.ancestor_pairs;
  v->tokens = reinterpret_cast<const int32_t*>(b + o[kTokens]);
  v->subtree_end = reinterpret_cast<const int32_t*>(b + o[kSubtreeEnd]);
  v->parent = reinterpret_cast<const int32_t*>(b + o[kParent]);
  v->depth = reinterpret_cast<const int32_t*>(b + o[kDepth]);
  v->node_id = reinterpret_cast<const int32_t*>(b + o[kNodeId]);
  v->child_off = reinterpret_cast<const int32_t*>(b + o[kChildOff]);
  v->child_pos = reinterpret_cast<const int32_t*>(b + o[kChildPos]);
  v->n_tokens = reinterpret_cast<const int32_t*>(b + o[kNTokens]);
  v->tok_base = reinterpret_cast<const int64_t*>(b + o[kTokBase]);
  v->node_info = reinterpret_cast<const int32_t*>(b + o[kNodeInfo]);
  v->n_nodes = reinterpret_cast<const int32_t*>(b + o[kNNodes]);
  v->seq_tree = reinterpret_cast<const int32_t*>(b + o[kSeqTree]);
  v->seq_off = reinterpret_cast<const int64_t*>(b + o[kSeqOff]);
  v->seq_pos = reinterpret_cast<const int32_t*>(b + o[kSeqPos]);
  return TPA_OK;
}

void tpa_tree_free(tpa_tree* tree) { delete tree; }

}  // extern "C"

uint64_t tpa_internal_blob_bytes(const tpa_tree* tree) { return tree ? tree->info.blob_bytes : 0; }
