/*
 * medusa.h -- C ABI of libmedusa_gb300.so, the GB300 (sm_103a) hot path of one
 * Medusa decode step.
 *
 * Sources, cited by page title and section:
 *   [MH] "Medusa Heads" glossary page (Ultralytics; Arabic and Portuguese
 *        editions), sections "How heads predict later tokens" and "Tree attention
 *        and acceptance".
 *   [SD] "Giai ma dau co: doan truoc roi kiem mot luot" (speculative-decoding
 *        e-book page), sections "Why a round always yields exactly k + 1 tokens"
 *        and "Faster without changing the result".
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless marked [host].  The caller owns every
 *     buffer; the library never allocates, frees or keeps a pointer after the
 *     call returns.
 *   - Device work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream).  Calls are asynchronous: no host synchronisation
 *     and no device-to-host copy happen inside them.
 *   - Tensors are dense row-major, in the shapes written next to them.  Weight
 *     matrices use the [out, in] layout of a linear layer's weight.  dtype
 *     MEDUSA_BF16 tensors hold bf16 values; MEDUSA_F32 tensors hold float.
 *     Vector loads need 16-byte aligned base pointers for weight, cache and logits
 *     tensors; a misaligned pointer returns MEDUSA_ERR_INVALID_ARG.
 *   - Return value: MEDUSA_OK (0), or a negative medusa_status with nothing
 *     enqueued.  medusa_last_error() returns a message for the calling thread's
 *     last failure.  A failed kernel launch returns MEDUSA_ERR_CUDA; errors raised
 *     by the device later surface in the caller's next CUDA synchronisation.
 *   - Kernels contain no traps, asserts or unbounded waits.  Device-resident
 *     values that break a precondition (out-of-range tokens, node indices or KV
 *     lengths) are clamped or skipped as each entry point documents.
 *   - Workspace: entry points that need scratch memory take `ws`/`ws_bytes`; the
 *     matching *_workspace() query returns the bytes needed for those shapes on the
 *     current device (it depends on the device's SM count).
 */
#ifndef MEDUSA_GB300_H
#define MEDUSA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MEDUSA_OK = 0,
    MEDUSA_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad alignment   */
    MEDUSA_ERR_UNSUPPORTED = -2, /* shape or dtype outside the supported limits  */
    MEDUSA_ERR_WORKSPACE = -3,   /* ws NULL or ws_bytes below the query's value  */
    MEDUSA_ERR_CUDA = -4,        /* a CUDA call or kernel launch failed          */
    MEDUSA_ERR_TIMEOUT = -5      /* a bounded device wait gave up (see below)    */
} medusa_status;

typedef enum { MEDUSA_F32 = 0, MEDUSA_BF16 = 1 } medusa_dtype;
typedef enum { MEDUSA_ACCEPT_GREEDY = 0, MEDUSA_ACCEPT_TYPICAL = 1 } medusa_accept_mode;

/* Message describing the calling thread's last failed call ("" if none). */
const char* medusa_last_error(void);

/* ABI version of this header (incremented on incompatible changes). */
int medusa_abi_version(void);

/* Device status of the tensor-core kernels (heads at bf16 batches 3-64, bf16
 * tree attention, the fused verification projection).  Their mbarrier waits
 * are bounded (about one second each).  A kernel whose wait gives up lets its
 * own copies and MMAs in flight complete, frees its tensor memory, marks the
 * outputs it owns (NaN attention rows, -1 top-k entries or -1 acceptance
 * outputs) and sets a status word on the device.  No kernel traps.
 *
 * medusa_device_status synchronises `stream`, then reads and clears the
 * current device's status words.  It returns MEDUSA_ERR_TIMEOUT if any wait on
 * that device gave up since the previous check (whatever stream the call was
 * on), MEDUSA_ERR_CUDA if the stream reported an error, MEDUSA_OK otherwise.
 * Unlike the other entry points it blocks the calling host thread. */
int medusa_device_status(void* stream);

/* Test hook: sets, on the current device, the limit in SM clock cycles of the
 * first waits of the tensor-core kernels (the waits for input tiles, MMA
 * results and free buffers); cycles <= 0 restores the default (2^31, about
 * one second).  The waits that let a giving-up kernel's copies and MMAs in
 * flight complete keep the default limit.  A limit of a few cycles makes the
 * waits run out on purpose, to exercise the path above.  Synchronous with
 * respect to the host; do not call it while kernels of the library run. */
int medusa_set_wait_limit(long long cycles);

/* ------------------------------------------------------------------------- */
/* 1. Medusa heads + per-head top-k  [MH, "How heads predict later tokens"]   */
/*                                                                           */
/* For each sequence b and head k (head k scores the token at t + k + 1):     */
/*   z      = h_b + SiLU(W1_k h_b + b1_k),  SiLU(x) = x * sigmoid(x)          */
/*   logits = W2_k z                                                          */
/* then the topk largest logits of each (b, k), sorted by value descending,   */
/* lowest token id first among equal values.  Accumulation is float32 and z   */
/* is kept in float32 whatever the storage dtype.                             */
/*   h        [B,H]      dtype    last hidden state                           */
/*   w1       [K,H,H]    dtype    row i = output feature i                    */
/*   b1       [K,H]      dtype                                                */
/*   w2       [K,V,H]    dtype    row v = token v                             */
/*   topk_idx [B,K,topk] int32    out                                         */
/*   topk_val [B,K,topk] float    out, may be NULL                            */
/*   logits   [B,K,V]    float    out, may be NULL (skips the write)           */
/* Limits: 1 <= K <= 64, 8 <= H <= 16384 with H % 8 == 0, topk <= 16,        */
/* topk <= V, and either 1 <= B <= 8 with B * H <= 49152 (any dtype), or      */
/* 9 <= B <= 64 for bf16 with H % 128 == 0.  Work is split over the vocab.    */
/* bf16 batches of 3 to 64 with H % 128 == 0 run on the tensor cores (z is    */
/* carried as three bf16 planes that hold 24 significant bits); h must then   */
/* be 16-byte aligned.  If a device-side wait gives up there (about one       */
/* second), the affected topk_idx entries are -1.                             */
/* ------------------------------------------------------------------------- */
size_t medusa_heads_topk_workspace(int B, int K, int H, int V, int topk);
int medusa_heads_topk(const void* h, const void* w1, const void* b1, const void* w2,
                      medusa_dtype dtype, int B, int K, int H, int V, int topk,
                      int32_t* topk_idx, float* topk_val, float* logits,
                      void* ws, size_t ws_bytes, void* stream);

/* Allocation-free variant of medusa_heads_topk (the pages have no counterpart:
 * this is a deployment convenience of this library).  Same arguments, results
 * and limits, minus ws/ws_bytes: the scratch comes from one device array of
 * MEDUSA_HEADS_STATIC_SCRATCH_BYTES (4 MiB) inside the library, for callers
 * that cannot call cudaMalloc -- e.g. an operator plugged into a host engine
 * that owns all device memory and gives its operators no workspace, or a
 * process whose device memory is fully reserved by a pool it may not grow.
 *   - Every GPU that loads the library holds that array until process exit.
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it with the
 *     unique ID of the current CUDA context; make that first call before any
 *     stream capture on the device.  A call in another context (after
 *     cudaDeviceReset, or in a context the caller created) looks the address
 *     up again, so that first call in the new context must also precede any
 *     capture.
 *   - Shapes whose scratch exceeds the maximum (e.g. large B*K*H) return
 *     MEDUSA_ERR_UNSUPPORTED without launching anything.
 *   - All calls share the one array: calls whose GPU work overlaps (other
 *     streams, other host threads on the same device) race and corrupt each
 *     other's results.  Serialize them, e.g. on one stream.
 *   - Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call. */
#define MEDUSA_HEADS_STATIC_SCRATCH_BYTES ((size_t)4 << 20)
int medusa_heads_topk_static(const void* h, const void* w1, const void* b1, const void* w2,
                             medusa_dtype dtype, int B, int K, int H, int V, int topk,
                             int32_t* topk_idx, float* topk_val, float* logits, void* stream);

/* ------------------------------------------------------------------------- */
/* 2. Candidate tree  [MH, "Tree attention and acceptance"]                   */
/*                                                                           */
/* A node is a tuple of ranks (r_1..r_d): rank r_k of head k's top-k list.    */
/* Its parent drops the last rank.  Canonical node order: root (the empty     */
/* tuple) first, then by depth, then lexicographic by rank tuple.             */
/* ------------------------------------------------------------------------- */

/* [host] The n_nodes - 1 most accurate rank tuples, accuracy of (r_1..r_d)
 * taken as prod_k head_p^k * rank_p^(r_k) (heads from 1, ranks from 0), larger
 * first; equal accuracy ties go to the shallower, then lexicographically smaller
 * tuple.  Tuples range over depths 1..max_depth (<= 16) and ranks
 * 0..max_rank-1.  paths_out [(n_nodes-1), max_depth], -1 padded, canonical
 * order.  Pure host code. */
int medusa_sparse_tree_paths(int n_nodes, int max_depth, int max_rank, double head_p,
                             double rank_p, int32_t* paths_out);

/* [host] Node table of the tree spanned by P rank tuples (every prefix of
 * every tuple is a node).  All arguments are host memory.
 *   rank_paths [P, max_depth] int32, -1 after the last rank
 *   parent/depth/rank [cap_nodes] out (rank = last rank of the tuple; -1 root)
 *   mask [cap_nodes * ceil(cap_nodes/64)] out: row i has W = ceil(N/64) words;
 *        bit m of row i is set iff node m is node i or one of its ancestors.
 *   retrieve [cap_paths, max_depth + 1] out: one row per leaf, leaves in node
 *        order, node indices root..leaf, -1 padded.  May be NULL.
 * Returns MEDUSA_ERR_INVALID_ARG when a tuple is malformed or capacity is short. */
int medusa_tree_layout(const int32_t* rank_paths, int P, int max_depth, int cap_nodes,
                       int cap_paths, int32_t* parent, int32_t* depth, int32_t* rank,
                       uint64_t* mask, int32_t* retrieve, int* N_out, int* W_out,
                       int* n_paths_out);

/* Candidate tokens: cand[b, 0] = root_tok[b] (the base model's own next token);
 * cand[b, i] = topk_idx[b, depth[i] - 1, rank[i]] for depth[i] >= 1.
 *   topk_idx [B,K,topk] int32; root_tok [B]; depth, rank [N] (node table);
 *   cand [B,N] int32 out.  A node whose depth or rank is out of range gets -1. */
int medusa_build_tree(const int32_t* topk_idx, const int32_t* root_tok, const int32_t* depth,
                      const int32_t* rank, int B, int K, int topk, int N, int32_t* cand,
                      void* stream);

/* ------------------------------------------------------------------------- */
/* 3. Tree attention  [MH, "Tree attention and acceptance"]                   */
/*                                                                           */
/* Every candidate is appended at once and sees only its tree ancestors: the  */
/* query of node i (sequence b, query head hq) attends to the prefix keys     */
/* [0, L_b) and to the tree keys at slots L_b + m for each m with bit m of    */
/* mask row i set:  out = softmax(scale * q.k) v, float32 softmax.            */
/*   q       [B,N,Hq,D]     dtype                                             */
/*   k_cache [B,Hkv,Lmax,D] dtype  tree keys already at slots [L_b, L_b+N)    */
/*   v_cache [B,Hkv,Lmax,D] dtype                                             */
/*   kv_len  [B] int32      L_b;  caller guarantees 0 <= L_b, L_b + N <= Lmax */
/*                          (out-of-range values are clamped into that range) */
/*   mask    [N, ceil(N/64)] uint64 from medusa_tree_layout                    */
/*   out     [B,N,Hq,D] float32                                               */
/* Query head hq reads KV head hq / (Hq / Hkv).  Limits: D in {64, 128},      */
/* 1 <= N <= 512, Hq % Hkv == 0, N * (Hq/Hkv) <= 4096; scale > 0 and finite   */
/* (MEDUSA_ERR_INVALID_ARG otherwise).                                        */
/* The bf16 path merges its KV-split partials on chip and needs no workspace: */
/* medusa_tree_attention_workspace returns 0 and ws may be NULL.  If a        */
/* device-side wait gives up (about one second), the affected outputs are NaN. */
/* ------------------------------------------------------------------------- */
size_t medusa_tree_attention_workspace(int B, int N, int Hq, int Hkv, int D, int Lmax);
int medusa_tree_attention(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* kv_len, const uint64_t* mask, medusa_dtype dtype,
                          int B, int N, int Hq, int Hkv, int D, int Lmax, float scale,
                          float* out, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* 4a. Tree acceptance  [MH, "Tree attention and acceptance"; SD, "Why a      */
/*     round always yields exactly k + 1 tokens"]                             */
/*                                                                           */
/* Row u of the verifier logits scores the token after node u.               */
/*  GREEDY:  candidate j passes iff cand[j] == argmax(row parent(j)), lowest  */
/*           token id on ties.                                                */
/*  TYPICAL: P = softmax(row / temperature), H = -sum P ln P,                 */
/*           tau = min(eps, delta * exp(-H)); candidate j passes iff          */
/*           P_parent(j)(cand[j]) > tau of row parent(j).  (The pages tie the  */
/*           threshold to the entropy without a formula; this is the form the */
/*           library uses.)  Softmax and entropy are float32.                 */
/* A node is accepted iff it and every ancestor pass (the root always is).    */
/* best = the deepest accepted node, lowest index on ties.  Outputs:          */
/*   accept_len [B]: depth(best) = accepted candidates (tokens = this + 1)    */
/*   best_node  [B]; path_nodes [B, Dmax+1]: root..best, -1 padded            */
/*   next_tok   [B]: argmax of row best (the correction / bonus token)       */
/*   logits [B,N,V] float32; cand [B,N]; parent, depth [N] from the layout.   */
/* Dmax = the tree's maximum depth.  Limits: N <= 512, V >= 1.               */
/* ------------------------------------------------------------------------- */
size_t medusa_verify_accept_workspace(int B, int N, int V);
int medusa_verify_accept_tree(const float* logits, const int32_t* cand, const int32_t* parent,
                              const int32_t* depth, int B, int N, int V, int Dmax,
                              medusa_accept_mode mode, float temperature, float eps,
                              float delta, int32_t* accept_len, int32_t* best_node,
                              int32_t* path_nodes, int32_t* next_tok, void* ws,
                              size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* 4b'. Typical acceptance with a sampled next token  [MH, "Tree attention    */
/*      and acceptance": in sampling, Medusa uses typical acceptance]         */
/*                                                                           */
/* accept_len, best_node and path_nodes as medusa_verify_accept_tree in      */
/* MEDUSA_ACCEPT_TYPICAL mode.  next_tok is drawn from P = softmax(row / T)   */
/* of the best node by the exponential race argmin_v -ln(U+_v) / w_v,         */
/* w_v = exp(row_v / T - max / T), lowest v on ties, with the random numbers  */
/* of 4b: key = f(f(f(f(f(seed) ^ 4) ^ b) ^ round) ^ 0) and U+_v taken from   */
/* next(key, v/2 + 1) as 4b states.  Workspace from                           */
/* medusa_verify_sample_workspace.                                            */
/* ------------------------------------------------------------------------- */
size_t medusa_verify_sample_workspace(int B, int N, int V);
int medusa_verify_accept_tree_sample(const float* logits, const int32_t* cand, const int32_t* parent,
                                     const int32_t* depth, int B, int N, int V, int Dmax,
                                     float temperature, float eps, float delta, uint64_t seed,
                                     uint64_t round, int32_t* accept_len, int32_t* best_node,
                                     int32_t* path_nodes, int32_t* next_tok, void* ws,
                                     size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* 4c. Verification projection fused with tree acceptance  [MH, "Tree         */
/*     attention and acceptance": the base model scores every branch of the   */
/*     tree in one pass]                                                      */
/*                                                                           */
/* Same outputs and rules as medusa_verify_accept_tree, but the verifier      */
/* logits are defined from the base model's last hidden state at each tree    */
/* node: logits[b,u,:] = lm_head . hidden_tree[b,u,:] (bf16 inputs, float32   */
/* accumulation).  The [B,N,V] logits are never written to memory: the       */
/* product runs on the tensor cores and is reduced tile by tile into per-row  */
/* argmax and softmax/entropy statistics.  Typical acceptance computes the    */
/* candidate logits it needs as separate float32 dot products.                */
/*   hidden_tree [B,N,H] bf16; lm_head [V,H] bf16 ([out, in]); 16-byte aligned */
/*   cand [B,N]; parent, depth [N]; outputs as in 4a.                         */
/* Limits: dtype MEDUSA_BF16; H % 8 == 0, H <= 65536; N <= 512; V <= 2^24.    */
/* If a device-side wait gives up (about one second), every output of the    */
/* call is -1.                                                               */
/* ------------------------------------------------------------------------- */
size_t medusa_verify_project_workspace(int B, int N, int H, int V);
int medusa_verify_project_tree(const void* hidden_tree, const void* lm_head, medusa_dtype dtype,
                               const int32_t* cand, const int32_t* parent, const int32_t* depth,
                               int B, int N, int H, int V, int Dmax, medusa_accept_mode mode,
                               float temperature, float eps, float delta, int32_t* accept_len,
                               int32_t* best_node, int32_t* path_nodes, int32_t* next_tok,
                               void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* 4b. Speculative-sampling acceptance along a chain of gamma drafts          */
/*     [SD, "Faster without changing the result"; "Why a round always yields  */
/*     exactly k + 1 tokens"]                                                  */
/*                                                                           */
/* Draft i (from 1) is accepted with probability min(1, p_i(x_i)/q_i(x_i)):   */
/* accepted iff u_i * q_i(x_i) < p_i(x_i), decided exactly.  At the first     */
/* rejection a token is drawn from max(0, p_i - q_i) normalised and the round */
/* ends; if all gamma are accepted a bonus token is drawn from p_{gamma+1}.   */
/* Random numbers (SplitMix64, Steele-Lea-Flood 2014; next(s, n) = n-th      */
/* output from state s, i.e. the mix of s + n * 0x9E3779B97F4A7C15):          */
/*   f(x) = next(x, 1);  key = f(f(f(f(f(seed) ^ stream) ^ b) ^ round) ^ pos)  */
/*   accept uniform of draft i (from 1): u_i = (next(key, 1) >> 40) / 2^24    */
/*     with stream 1, pos i.                                                  */
/*   race uniforms: output h_m = next(key, m + 1) serves two vocab entries:   */
/*     entry 2m uses bits 40..63 and entry 2m+1 uses bits 16..39 of h_m;      */
/*     U+_v = (those 24 bits + 1) / 2^24, in (0, 1].                          */
/*   A draw from weights w is the exponential race argmin_{w_v > 0}           */
/*   -ln(U+_v) / w_v (lowest v on ties): stream 2 pos i for the residual at   */
/*   rejected position i, stream 3 pos gamma+1 for the bonus; with no         */
/*   positive weight it falls back to the lowest v holding the largest p.     */
/*   p [B,gamma+1,V] float32; q [B,gamma,V] float32; draft [B,gamma] int32     */
/*   n_acc [B] out; out_tok [B,gamma+1] out: accepted drafts, then the drawn  */
/*   token, -1 padded (n_acc + 1 tokens).  gamma = 0 is allowed (q, draft may */
/*   be NULL).  Out-of-range draft tokens count as rejected.                  */
/* ------------------------------------------------------------------------- */
size_t medusa_verify_chain_workspace(int B, int gamma, int V);
int medusa_verify_accept_chain(const float* p, const float* q, const int32_t* draft, int B,
                               int gamma, int V, uint64_t seed, uint64_t round, int32_t* n_acc,
                               int32_t* out_tok, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------- */
/* 5. KV compaction  [MH, "Tree attention and acceptance": keep the longest   */
/*    accepted branch; its last hidden state feeds the heads next round]      */
/*                                                                           */
/* In place: for each b and i = 0..a (a = accept_len[b]) the K and V rows at  */
/* slot L_b + path_nodes[b,i] move to slot L_b + i for every KV head (all     */
/* rows are read before any is written, so overlapping moves are safe), then  */
/* kv_len[b] = L_b + a + 1.  h_next[b] = hidden_tree[b, best_node[b]].        */
/*   k_cache, v_cache [B,Hkv,Lmax,D] dtype (in/out); kv_len [B] (in/out)      */
/*   path_nodes [B,Dmax+1], accept_len [B], best_node [B]: from 4a            */
/*   hidden_tree [B,N,H] dtype and h_next [B,H] dtype: may both be NULL       */
/*   src_idx [B,Dmax+1] out, may be NULL: the source slot of each kept row,   */
/*   -1 padded.  A sequence whose accept_len, path or L_b is out of range is  */
/*   left unchanged and its src_idx row is set to -2.                         */
/* Limits: (D * element size) % 16 == 0; (Dmax + 1) * D * element size is at */
/* most 48 KB; B <= 65535.                                                   */
/* ------------------------------------------------------------------------- */
int medusa_kv_compact(void* k_cache, void* v_cache, int32_t* kv_len, const int32_t* path_nodes,
                      const int32_t* accept_len, const int32_t* best_node,
                      const void* hidden_tree, void* h_next, medusa_dtype dtype, int B, int Hkv,
                      int D, int Lmax, int N, int H, int Dmax, int32_t* src_idx, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MEDUSA_GB300_H */
