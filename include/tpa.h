/*
 * tpa.h — C ABI of libtpa, prefix-shared tree attention on GB300 (sm_103a).
 *
 * The method is "tree training" as described on the AReaL documentation page
 * "树训练" (tree training): sequences that share a prefix are packed into one
 * prefix trie so that every shared token is computed once; attention inside a
 * packed tree is causal with tree structure (a token attends only to its
 * ancestors and itself); log-probabilities are gathered back per original
 * sequence from the packed rows.
 *
 * Conventions for every call:
 *  - Every function returns an int status (TPA_OK = 0, negative = error) and
 *    never aborts or throws.  tpa_status_string() names a status.
 *  - The library owns only the host memory of a tpa_tree (freed by
 *    tpa_tree_free).  All device memory is allocated by the caller and passed
 *    as plain device pointers; the library allocates no device memory.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Device work is enqueued asynchronously on it; a launch failure
 *    is reported as TPA_ERR_CUDA by the call that launched it.  Kernel-side
 *    failures (a bounded wait that ran out) are recorded in a device status
 *    word and reported by tpa_sync_status().
 *  - Tensors are dense, row-major, with the layouts stated per call.
 *    bf16 means IEEE bfloat16 stored as uint16.
 */
#ifndef TPA_H_
#define TPA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* BLOCK_SIZE of the tree-training page (§注意力机制, FlexAttention block mask):
 * max_tokens_per_mb must be a multiple of it (§配置, note under the table). */
#define TPA_BLOCK_SIZE 128

enum tpa_status_code {
  TPA_OK = 0,
  TPA_ERR_INVALID_ARG = -1,        /* null pointer, bad size, bad alignment, unsupported shape */
  TPA_ERR_EMPTY_SEQUENCE = -2,     /* a sequence of length 0 */
  TPA_ERR_SEQ_TOO_LONG = -3,       /* a sequence longer than max_tokens_per_mb */
  TPA_ERR_NO_MEMORY = -4,          /* host allocation failed */
  TPA_ERR_CUDA = -5,               /* a CUDA runtime call or kernel launch failed */
  TPA_ERR_DEVICE_TIMEOUT = -6,     /* a kernel's bounded wait ran out (kernel returned early) */
  TPA_ERR_UNSUPPORTED_DEVICE = -7, /* current device is not compute capability 10.3 */
  TPA_ERR_BUFFER_TOO_SMALL = -8    /* a caller buffer is smaller than required */
};

/* ------------------------------------------------------------------------ */
/* Packing: tree training page, §树构建过程 steps 2-3 and §数据结构 TrieNode.  */
/* ------------------------------------------------------------------------ */

typedef struct tpa_tree tpa_tree; /* opaque; host memory owned by the library */

typedef struct {
  int32_t n_trees;            /* B: one tree per micro-batch */
  int32_t t_pad;              /* T_pad = max_tokens_per_mb (every tree padded to it) */
  int32_t n_seqs;             /* number of input sequences */
  int32_t max_nodes;          /* largest compressed-node count of any tree */
  int64_t total_seq_tokens;   /* sum of input lengths */
  int64_t total_tree_tokens;  /* sum over trees of real (non-pad) positions */
  int64_t total_nodes;        /* sum over trees of compressed nodes */
  int64_t ancestor_pairs;     /* sum over real positions of (depth + 1) */
  double tree_token_ratio;    /* total_tree_tokens / total_seq_tokens (§指标和监控) */
  uint64_t blob_bytes;        /* size of the metadata blob (host and device copies) */
  int32_t max_token;          /* largest token id of any sequence: a logits row must be wider */
  int32_t reserved_;
} tpa_tree_info;

/*
 * Per-tree flattened layout, as plain arrays inside one metadata blob.
 * The blob is built on the host by tpa_tree_pack; tpa_tree_upload copies it
 * verbatim into a caller device buffer; tpa_tree_make_view fills this struct
 * with pointers into either copy.  Position p of tree b lives at index
 * b * t_pad + p.  Positions are in preorder (§数据结构: nodes listed in
 * preorder; node tokens at inclusive [start_idx, end_idx]); positions
 * p >= n_tokens[b] are padding.
 */
typedef struct {
  int32_t n_trees, t_pad, n_seqs, max_nodes;
  int64_t total_seq_tokens;
  int64_t total_tree_tokens;
  int32_t max_token;          /* largest token id (the log-prob calls reject vocab <= max_token) */
  int32_t reserved_;
  int64_t ancestor_pairs;     /* sum over real positions of (depth + 1): sizes the backward's work items */
  const int32_t* tokens;      /* [B*T_pad] token id; pad -1 */
  const int32_t* subtree_end; /* [B*T_pad] E[p]: last position of the subtree of p's node;
                                 key p is visible to query i iff p <= i <= E[p]; pad -1 */
  const int32_t* parent;      /* [B*T_pad] position of the parent token; -1 under the root and at pad */
  const int32_t* depth;       /* [B*T_pad] number of ancestors = position id; pad 0 */
  const int32_t* node_id;     /* [B*T_pad] compressed node of p (tree-local, preorder); pad -1 */
  const int32_t* child_off;   /* [B*(T_pad+1)] CSR: children of p are child_pos[b*T_pad + child_off[b*(T_pad+1)+p] ..
                                 child_off[b*(T_pad+1)+p+1]) in ascending position order */
  const int32_t* child_pos;   /* [B*T_pad] child positions (tree-local); unused tail -1 */
  const int32_t* n_tokens;    /* [B] real positions per tree */
  const int64_t* tok_base;    /* [B+1] exclusive prefix sum of n_tokens (compact row numbering) */
  const int32_t* node_info;   /* [B*max_nodes*4] per node: start, end (inclusive), parent node (-1 under
                                 the root), subtree end; unused tail -1 */
  const int32_t* n_nodes;     /* [B] */
  const int32_t* seq_tree;    /* [n_seqs] tree holding each input sequence */
  const int64_t* seq_off;     /* [n_seqs+1] offsets of each sequence (same as the input offsets) */
  const int32_t* seq_pos;     /* [total_seq_tokens] tree position of every input token */
} tpa_tree_view;

/*
 * tpa_tree_pack — build the packed trees (tree training page, §树构建过程:
 * step 2 greedy first-fit-decreasing insertion into a trie, step 3 merging
 * linear chains into compressed nodes; §配置: each tree holds at most
 * max_tokens_per_mb tokens, a multiple of 128).
 *   tokens        [seq_offsets[n_seqs]] int32 token ids (>= 0), host memory
 *   seq_offsets   [n_seqs+1] int64, seq_offsets[0] = 0, non-decreasing, host
 *   n_seqs        >= 1
 *   max_tokens_per_mb  > 0 and a multiple of TPA_BLOCK_SIZE
 *   out           receives a new tree handle (set to NULL on error)
 * Rules: sequences are taken longest first (equal lengths in input order);
 * each goes into the first existing tree (creation order) whose token count
 * plus the sequence's unshared tokens fits, else into a new tree; a node
 * starts at a trie vertex whose parent is the root or branches, and extends
 * while the vertex has exactly one child; children are laid out in insertion
 * order.  Errors: TPA_ERR_INVALID_ARG, TPA_ERR_EMPTY_SEQUENCE,
 * TPA_ERR_SEQ_TOO_LONG, TPA_ERR_NO_MEMORY.  Host only; thread-safe.
 */
int tpa_tree_pack(const int32_t* tokens, const int64_t* seq_offsets, int32_t n_seqs,
                  int32_t max_tokens_per_mb, tpa_tree** out);

/*
 * tpa_extract_sequences — step 1 of §树构建过程 (提取序列): the real tokens of
 * each row of a padded batch are the input_ids entries whose attention_mask
 * entry is non-zero, in column order (left or right padding and interior
 * gaps alike).
 *   input_ids      [n_rows, row_len] int32 (host)
 *   attention_mask [n_rows, row_len] uint8, 0 = padding (host)
 *   tokens_out     host buffer of n_rows * row_len int32 (the first
 *                  offsets_out[n_rows] entries are written)
 *   offsets_out    [n_rows+1] int64 (written): row r is tokens
 *                  [offsets_out[r], offsets_out[r+1]) — the input format of
 *                  tpa_tree_pack.  A row without tokens gives an empty range.
 * Errors: TPA_ERR_INVALID_ARG.  Host only; thread-safe.
 */
int tpa_extract_sequences(const int32_t* input_ids, const uint8_t* attention_mask, int32_t n_rows,
                          int32_t row_len, int32_t* tokens_out, int64_t* offsets_out);

/* tpa_tree_pack on the sequences tpa_extract_sequences reads from a padded
 * batch (steps 1-3 of §树构建过程 in one call).  Arguments and errors as the
 * two calls; a row without tokens is TPA_ERR_EMPTY_SEQUENCE. */
int tpa_tree_pack_padded(const int32_t* input_ids, const uint8_t* attention_mask, int32_t n_rows,
                         int32_t row_len, int32_t max_tokens_per_mb, tpa_tree** out);

/* Sizes and counts of a packed tree set.  Errors: TPA_ERR_INVALID_ARG. */
int tpa_tree_get_info(const tpa_tree* tree, tpa_tree_info* info);

/* Host copy of the metadata blob (info.blob_bytes bytes, 256-byte aligned,
 * valid until tpa_tree_free).  NULL on a NULL tree. */
const void* tpa_tree_host_blob(const tpa_tree* tree);

/* Fill `view` with pointers into a blob copy starting at `base` (the host
 * blob or a device buffer written by tpa_tree_upload).  Pure pointer
 * arithmetic.  Errors: TPA_ERR_INVALID_ARG. */
int tpa_tree_make_view(const tpa_tree* tree, const void* base, tpa_tree_view* view);

/* Copy the host blob into `dev_blob` (a caller device buffer of at least
 * info.blob_bytes bytes, 256-byte aligned) on `stream` (cudaMemcpyAsync,
 * host-to-device).  The tree must stay alive until the copy has run.
 * Errors: TPA_ERR_INVALID_ARG, TPA_ERR_BUFFER_TOO_SMALL, TPA_ERR_CUDA. */
int tpa_tree_upload(const tpa_tree* tree, void* dev_blob, uint64_t dev_bytes, void* stream);

/* Release a tree handle (NULL is ignored). */
void tpa_tree_free(tpa_tree* tree);

/* ------------------------------------------------------------------------ */
/* Micro-batch / rank balancing: blog post "AReaL 序列打包算法 FFD 与 KK"
 * (FFD and KK sections, packing metrics).  Items with positive integer
 * weights — packed trees (weight = tree tokens or ancestor pairs) or
 * sequences (weight = length) — are split into groups: micro-batches of at
 * most `capacity`, or data-parallel ranks (a capacity larger than the total
 * makes the split purely about balance).  Host only; thread-safe.           */
/* ------------------------------------------------------------------------ */

enum { TPA_BALANCE_FFD = 0, TPA_BALANCE_KK = 1 };

/*
 * tpa_balance
 *   weights [n] int64 > 0, each <= capacity (host)
 *   capacity > 0: largest group weight
 *   min_groups >= 1, groups_divisor >= 1: the group count is >= min_groups
 *     and a multiple of groups_divisor
 *   algorithm TPA_BALANCE_FFD: items heaviest first (equal weights in input
 *     order); while fewer than min_groups groups exist an item opens a group,
 *     otherwise it joins the lightest group with room (equal loads: the
 *     earliest group), or opens a group when none has room; a group count
 *     that misses the rules raises min_groups to the next multiple of the
 *     divisor and the allocation is redone.  Groups are numbered in
 *     creation order.
 *   algorithm TPA_BALANCE_KK: k = max(min_groups, ceil(total / capacity))
 *     rounded up to the divisor; each item starts as a k-set partial
 *     partition; the two partitions of largest spread (max - min set sum;
 *     equal spreads: the older first) are merged by joining the i-th largest
 *     set of the first with the i-th smallest set of the second, until one
 *     remains.  Groups are numbered by final sum, heaviest first.  If a group
 *     exceeds the capacity the FFD result is returned instead.
 *   group_of [n] int32 (written): group of each item
 *   n_groups (written): number of groups
 *   algorithm_used (written if not NULL): the algorithm whose result this is
 * Errors: TPA_ERR_INVALID_ARG (null pointer, n < 1, non-positive argument or
 * weight, unknown algorithm, more groups required than items),
 * TPA_ERR_SEQ_TOO_LONG (a weight above the capacity), TPA_ERR_NO_MEMORY.
 */
int tpa_balance(const int64_t* weights, int32_t n, int64_t capacity, int32_t min_groups,
                int32_t groups_divisor, int32_t algorithm, int32_t* group_of, int32_t* n_groups,
                int32_t* algorithm_used);

/* Packing metrics of a grouping (the post's quality measures): group loads
 * L_g = sum of the weights in g; spread = max - min; mean = total / groups;
 * std_dev = population standard deviation of the loads; cv = std_dev / mean;
 * imbalance_ratio = max / mean; utilization = total / (groups * capacity);
 * wasted = groups * capacity - total (padding if every group is filled to
 * the capacity).  A group with no item has load 0. */
typedef struct {
  int32_t n_groups, pad_;
  int64_t total, max_load, min_load, spread, wasted;
  double mean, std_dev, cv, imbalance_ratio, utilization;
} tpa_packing_metrics_t;

/* Errors: TPA_ERR_INVALID_ARG (null pointer, n < 1, n_groups < 1, capacity
 * < 1, a group index outside [0, n_groups)), TPA_ERR_NO_MEMORY. */
int tpa_packing_metrics(const int64_t* weights, int32_t n, const int32_t* group_of, int32_t n_groups,
                        int64_t capacity, tpa_packing_metrics_t* out);

/* ------------------------------------------------------------------------ */
/* Block classification: tree training page, §树构建过程 step 4 (mask
 * generation) and §注意力机制 (block mask, BLOCK_SIZE 128, empty blocks are
 * skipped).  A 128x128 tile (query block qb, key block kb) is EMPTY when no
 * query in it sees any key in it, FULL when every query sees every key, and
 * PARTIAL otherwise.                                                        */
/* ------------------------------------------------------------------------ */

enum { TPA_BLOCK_EMPTY = 0, TPA_BLOCK_PARTIAL = 1, TPA_BLOCK_FULL = 2 };

typedef struct {
  int32_t n_trees, n_blk;     /* n_blk = T_pad / 128 */
  int32_t cap;                /* entries reserved per tree per CSR = n_blk*(n_blk+1)/2 */
  int32_t pad_;
  uint8_t* cls;               /* [B][n_blk][n_blk] class of (qb, kb) */
  int32_t* q_ptr;             /* [B][n_blk+1] CSR by query block (tree-local offsets) */
  int32_t* q_idx;             /* [B][cap] entries 2*kb + (FULL ? 1 : 0), ascending kb */
  int32_t* k_ptr;             /* [B][n_blk+1] CSR by key block */
  int32_t* k_idx;             /* [B][cap] entries 2*qb + (FULL ? 1 : 0), ascending qb */
  uint32_t* qmask;            /* [B][cap][128][4] for each PARTIAL entry e of q_idx: row r holds the
                                 visibility bits of query qb*128 + r (bit c of word c/32 = key
                                 kb*128 + c visible); FULL entries' rows are not written */
  uint32_t* sched;            /* [16] work counters of the attention kernels: zeroed by
                                 tpa_block_classify and left at zero by every attention call, so
                                 attention calls that use the same mask must not overlap on the GPU */
  int32_t* line_count;        /* [B][2][n_blk] scratch of tpa_block_classify: non-empty tiles per
                                 query block (row) and per key block (column) */
} tpa_blockmask_view;

/* Bytes of one device buffer holding a block mask for (n_trees, t_pad). */
uint64_t tpa_blockmask_bytes(int32_t n_trees, int32_t t_pad);

/* Slice a caller buffer of tpa_blockmask_bytes() bytes (256-byte aligned)
 * into a view.  Errors: TPA_ERR_INVALID_ARG. */
int tpa_blockmask_make_view(void* base, int32_t n_trees, int32_t t_pad, tpa_blockmask_view* view);

/* Classify every tile of every tree from the device subtree_end array and
 * build both CSR lists and the partial-tile bit rows (four kernels on `stream`).  `tree` must be a view of
 * the DEVICE blob; `mask` a view of a device buffer.  Integer only; results
 * are deterministic.  Errors: TPA_ERR_INVALID_ARG, TPA_ERR_CUDA. */
int tpa_block_classify(const tpa_tree_view* tree, const tpa_blockmask_view* mask, void* stream);

/* ------------------------------------------------------------------------ */
/* Dense ancestor mask: tree training page, §Megatron 引擎 (for gradient
 * checkpointing the Megatron engine passes a dense attention-mask tensor
 * instead of a BlockMask, since save_for_backward() serialises only
 * tensors).  M[b][i][j] = 1 iff key j is visible to query i, j <= i <= E[j];
 * pad rows and pad columns are 0.                                           */
/* ------------------------------------------------------------------------ */

enum { TPA_MASK_U8 = 0, TPA_MASK_BITS = 1 };

/* Bytes of a dense mask: B * T_pad^2 (TPA_MASK_U8) or B * T_pad^2 / 8
 * (TPA_MASK_BITS); 0 on invalid arguments. */
uint64_t tpa_dense_mask_bytes(int32_t n_trees, int32_t t_pad, int32_t format);

/*
 * tpa_dense_mask — write the dense mask of every tree.
 *   tree     view of the DEVICE blob
 *   out      device buffer of tpa_dense_mask_bytes() bytes, 16-byte aligned:
 *            TPA_MASK_U8   [B, T_pad, T_pad] uint8, out[b][i][j] = M[b][i][j]
 *            TPA_MASK_BITS [B, T_pad, T_pad / 32] uint32, bit (j % 32) of word
 *                          j / 32 of row i = M[b][i][j]
 *   invert   0: 1 marks a visible pair; 1: the complement (1 marks a removed
 *            pair, the convention of boolean masks whose True blocks attention)
 * One kernel on `stream`, bound by HBM writes.  Errors: TPA_ERR_INVALID_ARG,
 * TPA_ERR_BUFFER_TOO_SMALL, TPA_ERR_CUDA.
 */
int tpa_dense_mask(const tpa_tree_view* tree, void* out, uint64_t out_bytes, int32_t format, int32_t invert,
                   void* stream);

/* ------------------------------------------------------------------------ */
/* Tree attention (tree training page, §树构建过程 mask caption and
 * §注意力机制): for query position i of tree b and query head h,
 *   O_i = sum_{j: j <= i <= E[j]} softmax_j(scale * q_i . k_j) v_j
 * with key/value head h / (Hq / Hkv) (grouped-query attention) and
 * LSE_i = log sum_j exp(scale * q_i . k_j) (natural log).  Pad rows give
 * O = 0 and LSE = 0.  Computed in fp32 from bf16 inputs with an online
 * softmax on tcgen05 tensor cores; empty tiles are skipped and the ancestor
 * test runs only on partial tiles.                                          */
/* ------------------------------------------------------------------------ */

/*
 * tpa_tree_attn_fwd
 *   q [B, T_pad, Hq, d] bf16;  k, v [B, T_pad, Hkv, d] bf16 (device, 16-byte aligned;
 *     pad rows are read and must hold finite values)
 *   o [B, T_pad, Hq, d] bf16 (written);  lse [B, Hq, T_pad] fp32 (written)
 *   head_dim d in {64, 128};  Hq % Hkv == 0;  softmax_scale <= 0 selects 1/sqrt(d)
 * `tree` and `mask` are views of device buffers (mask filled by
 * tpa_block_classify for the same tree).  Errors: TPA_ERR_INVALID_ARG,
 * TPA_ERR_UNSUPPORTED_DEVICE, TPA_ERR_CUDA.
 */
int tpa_tree_attn_fwd(const tpa_tree_view* tree, const tpa_blockmask_view* mask,
                      const void* q, const void* k, const void* v, void* o, float* lse,
                      int32_t n_heads_q, int32_t n_heads_kv, int32_t head_dim,
                      float softmax_scale, void* stream);

/* Gradient output types of tpa_tree_attn_bwd. */
enum { TPA_GRAD_F32 = 0, TPA_GRAD_BF16 = 1 };

/* Workspace bytes needed by tpa_tree_attn_bwd: fp32 D = rowsum(dO * O)
 * [B, Hq, T_pad]; for TPA_GRAD_BF16 also fp32 staging rows for dK and dV
 * ([B, T_pad, Hkv, d] each, used by key tiles whose column is split into
 * several work items) and one 32-bit counter per (tree, kv head, key tile,
 * compute warp).  0 on invalid arguments. */
uint64_t tpa_tree_attn_bwd_workspace_bytes(int32_t n_trees, int32_t t_pad, int32_t n_heads_q,
                                           int32_t n_heads_kv, int32_t head_dim, int32_t grad_dtype);

/*
 * tpa_tree_attn_bwd — gradients of <dO, O> for the forward above:
 *   P_ij = exp(scale q_i.k_j - LSE_i), D_i = dO_i . O_i,
 *   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . v_j - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
 * dK/dV summed over the query heads of each key/value head.
 *   q, k, v, o, lse: as produced for / by tpa_tree_attn_fwd (o, lse read)
 *   dout [B, T_pad, Hq, d] bf16 (pad rows read, must be finite)
 *   dq [B, T_pad, Hq, d], dk, dv [B, T_pad, Hkv, d] (written; pad rows 0), fp32 for
 *     grad_dtype = TPA_GRAD_F32 or bf16 for TPA_GRAD_BF16.  Accumulation is fp32
 *     either way; fp32 outputs keep gradients of magnitude >= 8 within 2e-2 of
 *     the exact values, which a bf16 output (spacing 0.0625 there) cannot.
 *   workspace: device buffer of tpa_tree_attn_bwd_workspace_bytes() bytes,
 *     256-byte aligned, contents overwritten
 * dK/dV (per key tile) and dQ (per query tile) are accumulated in tensor
 * memory by separate kernels.  A key tile seen by more (query head, query
 * tile) pairs than one work item takes (a quarter of one SM's share of the
 * tree's steps, estimated from view.ancestor_pairs, at least 64) is split into
 * several items whose fp32 partial sums are added with atomic adds, into the
 * dK/dV rows for fp32 gradients or into workspace rows that the last item
 * converts to bf16; those rows can differ in the last bits between calls.
 * Every other output is deterministic.
 * Errors: as tpa_tree_attn_fwd, plus TPA_ERR_BUFFER_TOO_SMALL.
 */
int tpa_tree_attn_bwd(const tpa_tree_view* tree, const tpa_blockmask_view* mask,
                      const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv,
                      void* workspace, uint64_t workspace_bytes,
                      int32_t n_heads_q, int32_t n_heads_kv, int32_t head_dim,
                      float softmax_scale, int32_t grad_dtype, void* stream);

/*
 * tpa_tree_attn_bwd_noalloc — tpa_tree_attn_bwd for callers that cannot
 * provide a device workspace.  The tree-training pages have no counterpart;
 * this is a deployment variant.  Runtimes that reserve the whole device for
 * their own memory pool (and forbid further cudaMalloc calls), or plain-C
 * callers with no allocator at hand, cannot hand the library a workspace, so
 * this call takes its scratch from a fixed 16 MiB array compiled into the
 * library instead.  Every GPU that loads the library holds that array until
 * the process exits.
 *   Arguments: as tpa_tree_attn_bwd, without workspace / workspace_bytes.
 *   Limit: the scratch of tpa_tree_attn_bwd_workspace_bytes() must fit in
 *     16 MiB: B * T_pad * Hq * 4 bytes for fp32 gradients (e.g. 8 trees of
 *     8192 tokens with 64 query heads), plus B * T_pad * Hkv * d * 8 bytes and
 *     the counters for bf16 gradients (e.g. 2 trees of 8192 tokens with 32
 *     query and 2 kv heads of d 128).  Larger problems return
 *     TPA_ERR_BUFFER_TOO_SMALL and enqueue nothing.
 *   Allocation: none (no cudaMalloc, no cudaFree, no allocating library call).
 *   Set-up: the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress with that device current) and caches it; make that
 *     first call before any stream capture.  The cached address belongs to the
 *     device's current context: after cudaDeviceReset (or anything else that
 *     destroys the primary context) it is stale, so do not call this entry
 *     point on that device again in the same process.
 *   Sharing: every call on a device uses the same array, which keeps the last
 *     call's contents (each call rewrites all of the scratch it reads, so
 *     nothing carries over).  Calls that overlap on the GPU — on different
 *     streams, or from several host threads without ordering — race on it and
 *     must be serialised by the caller.
 * Errors: as tpa_tree_attn_bwd.
 */
int tpa_tree_attn_bwd_noalloc(const tpa_tree_view* tree, const tpa_blockmask_view* mask,
                              const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int32_t n_heads_q, int32_t n_heads_kv, int32_t head_dim,
                              float softmax_scale, int32_t grad_dtype, void* stream);

/* ------------------------------------------------------------------------ */
/* Log-probabilities and entropy (tree training page, §对数概率计算): labels
 * cannot come from rolling input_ids; each tree row is processed once (the
 * node-level cache) and the within-node and node-to-child transition labels
 * of that row are gathered in the same pass; results are then regathered
 * per original sequence.                                                   */
/* ------------------------------------------------------------------------ */

enum { TPA_LOGITS_COMPACT = 0, TPA_LOGITS_PADDED = 1 };

/*
 * tpa_tree_logprobs_entropy
 *   logits   bf16 rows of width `vocab`, device; row of (tree b, position p) is
 *            tok_base[b] + p (TPA_LOGITS_COMPACT) or b * T_pad + p
 *            (TPA_LOGITS_PADDED); consecutive rows `row_stride` elements apart
 *            (row_stride >= vocab, multiple of 8; base 16-byte aligned)
 *   pos_logp    [B*T_pad] fp32: at position c with parent r,
 *               log_softmax(logits[row r])[token c]; 0 under the root and at pad
 *   pos_entropy [B*T_pad] fp32: -sum_v p_v log p_v of row p (natural log); 0 at pad
 *   seq_logp    [total_seq_tokens] fp32: for sequence s at token t,
 *               pos_logp[next position of s] (t < L-1) and 0 at t = L-1
 *   seq_entropy [total_seq_tokens] fp32: pos_entropy at each token of s
 * All outputs are device buffers and are written completely.  Every token id
 * of the tree must be below `vocab`: a view whose max_token is >= vocab is
 * refused (TPA_ERR_INVALID_ARG) before any launch.  Should a label still fall
 * outside the row (a view edited by hand), the kernel does not read it: that
 * position's log-prob is NaN and the next tpa_sync_status() returns
 * TPA_ERR_INVALID_ARG.  Logits of -inf (masked vocabulary entries) are
 * allowed: they add nothing to the entropy (p log p -> 0 as p -> 0), and a
 * label at such an entry gets a log-prob of -inf; a row whose logits are all
 * -inf (or all below -1e30) has no distribution and gives NaN.  Errors:
 * TPA_ERR_INVALID_ARG,
 * TPA_ERR_CUDA.
 */
int tpa_tree_logprobs_entropy(const tpa_tree_view* tree, const void* logits, int64_t row_stride,
                              int32_t layout, int32_t vocab, float* pos_logp, float* pos_entropy,
                              float* seq_logp, float* seq_entropy, void* stream);

/*
 * tpa_lm_head_logprobs_entropy — the log-prob pass above with the LM head
 * fused in front of it (the step upstream of §对数概率计算): the logits of
 * compact tree row r are logits[r, v] = sum_k hidden[r, k] * weight[v, k],
 * computed tile by tile on tcgen05 tensor cores (bf16 inputs, fp32
 * accumulation) and consumed in place, so no logits tensor is written.
 * Outputs and their definitions are those of tpa_tree_logprobs_entropy.
 *   hidden   [total_tree_tokens, hidden_size] bf16, device, 16-byte aligned;
 *            row tok_base[b] + p is tree b, position p (compact rows)
 *   weight   [vocab, hidden_size] bf16, device, 16-byte aligned
 *   hidden_size a multiple of 64, <= 65536;  vocab >= 1;  every token id of the
 *            tree must be < vocab (a view whose max_token is >= vocab is
 *            refused with TPA_ERR_INVALID_ARG; a larger id in a view edited
 *            by hand yields NaN at its position)
 *   workspace device buffer of tpa_lm_head_workspace_bytes() bytes, 256-byte
 *            aligned, contents overwritten (per-row softmax partials, label
 *            logits, a work counter)
 * Kernels on `stream`: the fused GEMM + statistics kernel, a combine kernel
 * and the per-sequence gather.  Errors: TPA_ERR_INVALID_ARG,
 * TPA_ERR_BUFFER_TOO_SMALL, TPA_ERR_CUDA.
 */
uint64_t tpa_lm_head_workspace_bytes(int64_t rows, int32_t vocab, int32_t n_trees, int32_t t_pad);
int tpa_lm_head_logprobs_entropy(const tpa_tree_view* tree, const void* hidden, const void* weight,
                                 int32_t hidden_size, int32_t vocab, void* workspace,
                                 uint64_t workspace_bytes, float* pos_logp, float* pos_entropy,
                                 float* seq_logp, float* seq_entropy, void* stream);

/* ------------------------------------------------------------------------ */
/* Status                                                                    */
/* ------------------------------------------------------------------------ */

/* Synchronize `stream`, then read and clear the device status words of all
 * kernels: TPA_OK, TPA_ERR_DEVICE_TIMEOUT (a bounded wait ran out),
 * TPA_ERR_INVALID_ARG (a kernel met an input outside its range, such as a
 * label id >= vocab, and skipped it) or TPA_ERR_CUDA. */
int tpa_sync_status(void* stream);

/* Diagnostic for the bounded waits above: launches one thread on `stream`
 * that waits on a shared-memory mbarrier with the same clock-bounded wait the
 * attention kernels use (`limit_ns` in nanoseconds, counted in SM cycles at no
 * more than 2.1 GHz, so the real bound is at least that long).  arrive != 0:
 * the thread completes the barrier's phase first and the wait succeeds;
 * arrive == 0: nothing arrives, the wait runs out and sets the device status
 * word, so the next tpa_sync_status() returns TPA_ERR_DEVICE_TIMEOUT (and
 * clears it).  No fault or hang is involved: the kernel returns either way.
 * Errors: TPA_ERR_INVALID_ARG (limit_ns 0 or above 10 s), TPA_ERR_CUDA. */
int tpa_wait_probe(uint64_t limit_ns, int32_t arrive, void* stream);

/* TPA_OK when the current CUDA device is compute capability 10.3 (sm_103),
 * TPA_ERR_UNSUPPORTED_DEVICE otherwise, TPA_ERR_CUDA without a device. */
int tpa_device_check(void);

/* Static, human-readable name of a status code. */
const char* tpa_status_string(int status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int tpa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TPA_H_ */
