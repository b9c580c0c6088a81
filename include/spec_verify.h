/*
 * spec_verify.h -- C ABI of the batched draft-token verification library (GB300, sm_103a).
 *
 * One speculative-decoding round ends with a target forward over the gamma drafted
 * positions plus one; this library takes those target logits, the drafter's logits and
 * tokens, and decides what is kept. Sources, by page title and section:
 *
 *   [SpS] speculative-sampling article ("大模型推理的投机采样：Draft 小模型辅助与验证加速"),
 *         section "核心算法数学原理：无损拒绝采样": a draft token x is accepted when a uniform
 *         r satisfies r <= min(1, p(x)/q(x)); at the first rejection a replacement is drawn
 *         from max(0, p - q)/norm and the remaining drafts are dropped; section "核心实现":
 *         the target scores the last gamma+1 positions.
 *   [CoD] "Chain of Draft" article, section 3.2: NKL = KL(draft || target) / log(vocab),
 *         both rows softmaxed at one temperature, drafts kept while NKL < delta (0.15).
 *   [MTP] Gemma 4 multi-token-prediction drafter article, section 2.3: greedy verification
 *         (accept while the draft equals the target argmax; the target's argmax replaces
 *         the first mismatch).
 *   [PD]  Parallel Drafting article, section 2.2: the P-EAGLE draft tree (three root
 *         candidates, at most 12 nodes), verified along its longest accepted path.
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer unless its comment says "host".
 *     The caller owns every buffer; the library keeps no pointer after the call returns
 *     and allocates no memory.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *     stream) and is asynchronous. The return value reports only what can be checked
 *     on the host before launch (null pointers, sizes, temperature, dtype, workspace
 *     size) and launch failures; it never waits for the GPU.
 *   - Data errors found on the GPU are OR-ed into *device_status (a 32-bit device word,
 *     SPEC_DEV_* bits). The word is sticky: the library never clears it, the caller
 *     zeroes it when it wants a fresh reading. A sequence with a data error reports
 *     n = -1, -1 in its integer outputs and NaN in its real outputs. No kernel traps
 *     or asserts; every wait (the sampler polling a sequence's decision, a warp of the
 *     multi-draft pair pass over misaligned rows waiting for its bulk copies) is bounded
 *     and reports SPEC_DEV_TIMEOUT if it runs out.
 *   - Logits are row-major [rows, V] with V contiguous, fp32 or bf16 (raw bf16 bit
 *     patterns). Rows whose byte size is a multiple of 16 and whose base pointers are
 *     16-byte aligned take the vectorised path. Any other layout takes the phased
 *     vector path (each tile applies its row's offset within the 16-byte grid; row pairs
 *     whose two rows sit at different offsets have the draft's vectors shifted to the
 *     target's), with the same results: it reads whole aligned 16-byte blocks, so it may
 *     read up to 15 bytes before a row's first or after its last element, always inside
 *     a 16-byte block that holds one of the row's elements (never used, never written).
 *   - Every pointer is aligned to its element type: logits to 2 (bf16) or 4 (fp32)
 *     bytes, int32 and float arrays to 4, the statistics block and double outputs to 8.
 *     A misaligned pointer is SPEC_ERR_INVALID_ARG.
 *   - Packed batches: sequence b has gamma_b drafts. Its draft rows, draft tokens and
 *     u_accept entries start at cu_draft[b]; its target rows (gamma_b + 1 of them: one
 *     per draft plus the bonus row) and its out_tokens entries start at cu_draft[b] + b.
 *     cu_draft == NULL means a dense batch with gamma_b = gamma for every b.
 *   - `workspace` is scratch memory of at least spec_workspace_bytes() bytes, 256-byte
 *     aligned. Its contents need no initialisation and are meaningless between calls.
 *     Two calls may not use one workspace at the same time (e.g. on two streams).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* spec_stream_t; /* the same handle as cudaStream_t */

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1, /* null pointer, bad size, non-finite or non-positive T, bad tree */
  SPEC_ERR_DTYPE = 2,       /* unknown spec_dtype */
  SPEC_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than spec_workspace_bytes() */
  SPEC_ERR_CUDA = 6,        /* a CUDA call or kernel launch failed */
  SPEC_ERR_TOO_LARGE = 7    /* spec_verify_stochastic_static: the problem needs more scratch than it has */
} spec_status;

/* bits of *device_status */
#define SPEC_DEV_TOKEN_RANGE 1u /* a draft or node token outside [0, V) ([PD] section 4.1: token ids must agree) */
#define SPEC_DEV_NONFINITE 2u   /* a NaN or infinite logit in a row the sequence uses */
#define SPEC_DEV_OFFSETS 4u     /* cu_draft not non-decreasing from 0 to total_draft, or a gamma_b > gamma */
#define SPEC_DEV_TIMEOUT 8u     /* an internal wait gave up (bounded waits); the affected sequences are undecided */
#define SPEC_DEV_POSITION 16u   /* spec_options.position[b] < 1 */
#define SPEC_DEV_BOUNDS 32u     /* only in a library built with SPEC_BOUNDS_CHECK=1: a computed memory access fell
                                   outside its buffer (that access was skipped); never set by the ordinary build */

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* which call a workspace is sized for */
typedef enum { SPEC_MODE_STOCHASTIC = 0, SPEC_MODE_GREEDY = 1, SPEC_MODE_NKL = 2 } spec_mode;

#define SPEC_MAX_GAMMA 128    /* largest gamma_b */
#define SPEC_MAX_TREE_NODES 64

/* Batch geometry, passed by value. */
typedef struct {
  int32_t B;               /* sequences, >= 0 (0 = nothing to do) */
  int32_t gamma;           /* dense: drafts per sequence; packed: an upper bound on every gamma_b; 0..SPEC_MAX_GAMMA */
  int32_t V;               /* vocabulary size, >= 1 */
  int32_t total_draft;     /* sum of gamma_b (dense: B * gamma); must equal cu_draft[B] */
  const int32_t* cu_draft; /* device [B+1], non-decreasing prefix sums of gamma_b; NULL = dense */
} spec_batch;

/* Bytes of scratch memory a call of `mode` needs for geometry g and element type dtype
 * (0 for an invalid geometry or dtype). The workspace must be 256-byte aligned. */
size_t spec_workspace_bytes(spec_batch g, spec_dtype dtype, spec_mode mode);

/* Bytes of scratch memory spec_verify_tree needs (256-byte aligned, as above). */
size_t spec_tree_workspace_bytes(int32_t B, int32_t N, int32_t V);

/*
 * Stochastic verification with residual resampling and a bonus token ([SpS]), with the
 * per-position NKL of [CoD] 3.2 and the greedy decision of [MTP] 2.3 from the same read.
 *
 * For each sequence b and position i < gamma_b, with p = softmax(target row i / T) and
 * q = softmax(draft row i / T), x_i = draft_tokens[i]:
 *   alpha_i = min(1, p(x_i) / q(x_i)); draft i is accepted iff u_accept[i] <= alpha_i;
 *   n = the first i not accepted, else gamma_b;
 *   if n < gamma_b the last token is the smallest y with C(y) > u_sample[b] * Z, C the
 *   running sum in token order of max(0, p - q) over row pair n and Z its total;
 *   if n == gamma_b the same rule over p of target row gamma_b (the bonus token).
 *   (Z == 0 at a rejection, reachable only through rounding: the row p is used instead.)
 *
 *   target_logits [total_draft + B, V], draft_logits [total_draft, V], draft_tokens
 *   [total_draft] int32, u_accept [total_draft] fp32 in [0,1), u_sample [B] fp32 in [0,1),
 *   temperature: finite, > 0, applied to both rows. Uniforms are used as given: a u_accept
 *   above 1 rejects its draft whatever alpha is.
 * Outputs (caller-allocated):
 *   n_accepted [B]                     required: n per sequence (-1 on a data error)
 *   out_tokens [total_draft + B]       required: per sequence x_0..x_{n-1}, then the
 *                                      correction or bonus token, then -1 up to gamma_b
 *   p_x, q_x, alpha [total_draft]      optional (NULL skips): p(x_i), q(x_i), alpha_i
 *   nkl [total_draft], nkl_mask [total_draft]  optional: KL(q||p)/ln V and (nkl < nkl_delta)
 *   greedy_n [B], greedy_tokens [total_draft + B]  optional: the greedy decision on the
 *                                      same target rows (argmax of the raw logits, ties to
 *                                      the lowest id), laid out like n_accepted / out_tokens
 *   device_status [1]                  required, sticky (see above)
 */
spec_status spec_verify_stochastic(spec_batch g, spec_dtype dtype, const void* target_logits,
                                   const void* draft_logits, const int32_t* draft_tokens,
                                   float temperature, const float* u_accept, const float* u_sample,
                                   int32_t* n_accepted, int32_t* out_tokens, float* p_x, float* q_x,
                                   float* alpha, float* nkl, uint8_t* nkl_mask, float nkl_delta,
                                   int32_t* greedy_n, int32_t* greedy_tokens, uint32_t* device_status,
                                   void* workspace, size_t workspace_bytes, spec_stream_t stream);

/*
 * Greedy argmax-match verification ([MTP] 2.3): g_i = argmax of target row i (raw logits,
 * ties to the lowest id); n = the first i with draft_tokens[i] != g_i, else gamma_b;
 * out = x_0..x_{n-1}, g_n, then -1 up to gamma_b. Reads the target rows only.
 *   target_logits [total_draft + B, V], draft_tokens [total_draft];
 *   n_accepted [B], out_tokens [total_draft + B], device_status [1].
 */
spec_status spec_verify_greedy(spec_batch g, spec_dtype dtype, const void* target_logits,
                               const int32_t* draft_tokens, int32_t* n_accepted, int32_t* out_tokens,
                               uint32_t* device_status, void* workspace, size_t workspace_bytes,
                               spec_stream_t stream);

/*
 * Greedy tree verification ([PD] 2.2). Every sequence carries the same tree of N nodes.
 *   parent: HOST [N], parent[j] in {-1, 0..j-1} (-1 = a root); 1 <= N <= SPEC_MAX_TREE_NODES.
 *   target_logits [B * (N + 1), V]: row 0 of a sequence scores the position before the
 *   tree, row j+1 scores the position after node j. node_tokens [B, N] int32.
 * Node j is accepted iff node_tokens[j] equals the argmax of its parent's row (row 0 for a
 * root) and its parent is accepted. The pick is the accepted node of greatest depth (ties
 * to the lowest node index). With D = spec_tree_depth(parent, N):
 *   accept_len [B]           depth of the pick (0 if no node is accepted)
 *   path_nodes [B, D]        node indices from the root to the pick, then -1
 *   out_tokens [B, D + 1]    the path's tokens, then the argmax of the pick's row (of row 0
 *                            if none), then -1
 * A data error gives accept_len = -1 and -1 everywhere in that sequence's outputs.
 */
spec_status spec_verify_tree(int32_t B, int32_t N, int32_t V, spec_dtype dtype, const void* target_logits,
                             const int32_t* node_tokens, const int32_t* parent, int32_t* accept_len,
                             int32_t* path_nodes, int32_t* out_tokens, uint32_t* device_status,
                             void* workspace, size_t workspace_bytes, spec_stream_t stream);

/* Depth of the tree described by the HOST array parent[N] (a root has depth 1); -1 if the
 * array is not a valid topologically ordered forest or N is out of range. */
int32_t spec_tree_depth(const int32_t* parent, int32_t N);

/*
 * NKL alone ([CoD] 3.2) for every (target row i, draft row i), i < gamma_b:
 *   nkl[i] = KL(q || p) / ln V with q = softmax(draft/T), p = softmax(target/T), natural log,
 *   unclamped; nkl_mask[i] = (nkl[i] < delta), optional (NULL skips).
 * Layout as spec_verify_stochastic (target row i of sequence b at cu_draft[b] + b + i).
 * A non-finite logit in a row pair gives NaN / 0 for that pair only.
 */
spec_status spec_nkl(spec_batch g, spec_dtype dtype, const void* target_logits, const void* draft_logits,
                     float temperature, float delta, float* nkl, uint8_t* nkl_mask,
                     uint32_t* device_status, void* workspace, size_t workspace_bytes,
                     spec_stream_t stream);

/*
 * Policy variants: each *_ex call takes every argument of the plain call plus `options`
 * (a HOST pointer, read during the call; NULL = the plain call). Zero-initialise the
 * struct and set what is used; fields a call does not use are ignored.
 */
#define SPEC_STATS_SLOTS 64

/* One time bucket of acceptance statistics. */
typedef struct {
  int64_t bucket;    /* the caller's label of the bucket this slot holds */
  uint64_t rounds;   /* sequences with gamma_b > 0 and no data error verified in it */
  uint64_t accepted; /* their accepted drafts, sum of n_b */
  uint64_t drafted;  /* their drafts, sum of gamma_b */
  uint64_t rate_fx;  /* sum of n_b / gamma_b, each rounded to a multiple of 2^-32, in units of 2^-32 */
  uint64_t rate2_fx; /* sum of (n_b / gamma_b)^2, likewise */
} spec_stats_slot;

/* Device-resident acceptance statistics ([MTP] 5.1: accepted drafts per round; [PD] 5.2:
 * the standard deviation of the acceptance rate over a window, ARSD): a ring in which
 * bucket k lives in slot k mod SPEC_STATS_SLOTS. Zero-fill it once before first use. */
typedef struct {
  spec_stats_slot slot[SPEC_STATS_SLOTS];
} spec_accept_stats;

typedef struct {
  /* stochastic: > 0 and finite = the temperature T_d the drafts were drawn at ([PD] 4.4:
   * draft 0.3-0.5, target 0.7-0.9). q = softmax(draft / T_d) for q(x), alpha and the
   * residual; NKL still scales both rows by the target temperature ([CoD] 3.2), so a call
   * that asks for nkl or nkl_mask sums each draft row at both temperatures (one more
   * exponential per draft logit), and one that asks for neither does not.
   * 0 = T_d equals the target temperature. */
  float temperature_draft;
  /* stochastic, NKL: device [B] or NULL. The 1-based position of each sequence's first
   * draft in the generated text; the NKL mask of draft i then compares against
   * delta_pos = min(delta_max, delta * (1 + delta_alpha * log2(position[b] + i)))
   * ([CoD] 4.3; the page's values 0.08 and 0.3). A position < 1 sets
   * SPEC_DEV_POSITION and masks that sequence's drafts out (mask 0); its other outputs
   * are unaffected. */
  const int32_t* position;
  float delta_alpha;
  float delta_max;
  /* stochastic, greedy: > 0 enables block-accept ([CoD] 3.3; the page's value is 3):
   * block_n [B] gets e, the end of the longest run of >= min_block_len consecutive
   * positions where the draft equals the target argmax (the earliest of equally long
   * runs), or 0 when there is none (-1 on a data error); block_tokens [total_draft] gets
   * the draft tokens before e and the target argmax from e on. Either may be NULL when it
   * has no elements (B = 0, or total_draft = 0). */
  int32_t min_block_len;
  int32_t* block_n;
  int32_t* block_tokens;
  /* stochastic, greedy: device statistics or NULL. Every sequence with gamma_b > 0 and no
   * data error adds one round to the slot of stats_bucket, which is first reset if it
   * holds another bucket. Bucket labels must not decrease from call to call. */
  spec_accept_stats* stats;
  int64_t stats_bucket;
} spec_options;

spec_status spec_verify_stochastic_ex(spec_batch g, spec_dtype dtype, const void* target_logits,
                                      const void* draft_logits, const int32_t* draft_tokens,
                                      float temperature, const float* u_accept, const float* u_sample,
                                      int32_t* n_accepted, int32_t* out_tokens, float* p_x, float* q_x,
                                      float* alpha, float* nkl, uint8_t* nkl_mask, float nkl_delta,
                                      int32_t* greedy_n, int32_t* greedy_tokens, const spec_options* options,
                                      uint32_t* device_status, void* workspace, size_t workspace_bytes,
                                      spec_stream_t stream);

spec_status spec_verify_greedy_ex(spec_batch g, spec_dtype dtype, const void* target_logits,
                                  const int32_t* draft_tokens, int32_t* n_accepted, int32_t* out_tokens,
                                  const spec_options* options, uint32_t* device_status, void* workspace,
                                  size_t workspace_bytes, spec_stream_t stream);

spec_status spec_nkl_ex(spec_batch g, spec_dtype dtype, const void* target_logits, const void* draft_logits,
                        float temperature, float delta, float* nkl, uint8_t* nkl_mask,
                        const spec_options* options, uint32_t* device_status, void* workspace,
                        size_t workspace_bytes, spec_stream_t stream);

/*
 * Summary of the statistics over the buckets (bucket_now - window, bucket_now],
 * 1 <= window <= SPEC_STATS_SLOTS, written to out [6] (device, fp64): rounds, accepted
 * drafts, drafts, mean accepted drafts per round, mean acceptance rate (n_b / gamma_b),
 * and ARSD, the population standard deviation of the per-round acceptance rates
 * (0 when there is no round).
 */
spec_status spec_accept_summary(const spec_accept_stats* stats, int64_t bucket_now, int32_t window, double* out,
                                spec_stream_t stream);

/*
 * Multi-draft verification ([MTP] 6.2: several drafters each propose a draft, the target
 * verifies all of them and the longest accepted path is kept; [CoD] 4.4: the pairwise NKL
 * matrix of the drafts, consensus below 0.1 and divergence above 0.15).
 *
 * G groups of K candidate sequences, each with gamma drafts, laid out as a dense batch of
 * G*K sequences (candidate k of group g is sequence g*K + k): target_logits
 * [G*K*(gamma+1), V], draft_logits [G*K*gamma, V], draft_tokens [G*K*gamma]. Every
 * candidate is verified as by spec_verify_stochastic (stochastic != 0; u_accept
 * [G*K*gamma], u_sample [G*K]) or spec_verify_greedy (stochastic == 0; the uniforms
 * are not read). Outputs:
 *   n_accepted [G*K], out_tokens [G*K*(gamma+1)]   every candidate's result
 *   best_k [G], best_n [G], best_tokens [G*(gamma+1)]  the kept candidate: the most
 *                                      accepted drafts, the lowest k among equals (-1
 *                                      when every candidate of the group had a data
 *                                      error). With stochastic verification this choice
 *                                      does not preserve the target distribution.
 *   pair_nkl [G*gamma*K*K]             optional: at draft position i of group g,
 *                                      M[a][b] = KL(q_a || q_b) / ln V between the
 *                                      candidates' draft rows i, q = softmax(row / T);
 *                                      zero diagonal; NaN for a non-finite row
 *   consensus, divergence [G*gamma]    optional: some pair a != b below consensus_nkl in
 *                                      both directions; every entry off the diagonal
 *                                      above divergence_nkl
 * 2 <= K <= SPEC_MAX_CANDIDATES. Rows on the 16-byte grid (V * element size a multiple of 16,
 * 16-byte aligned bases) are read once: one pass verifies the K candidates of a position and
 * fills their matrix. Rows off the grid are verified by the batch kernels and the draft rows
 * are then read a second time for the matrix.
 */
#define SPEC_MAX_CANDIDATES 4

typedef struct {
  int32_t G;     /* groups, >= 0 */
  int32_t K;     /* candidates per group, 2..SPEC_MAX_CANDIDATES */
  int32_t gamma; /* drafts per candidate, 0..SPEC_MAX_GAMMA */
  int32_t V;     /* vocabulary size, >= 1 */
} spec_multi_batch;

size_t spec_multi_workspace_bytes(spec_multi_batch m, spec_dtype dtype, int32_t stochastic);

spec_status spec_verify_multi(spec_multi_batch m, spec_dtype dtype, int32_t stochastic, const void* target_logits,
                              const void* draft_logits, const int32_t* draft_tokens, float temperature,
                              const float* u_accept, const float* u_sample, float consensus_nkl,
                              float divergence_nkl, int32_t* n_accepted, int32_t* out_tokens, int32_t* best_k,
                              int32_t* best_n, int32_t* best_tokens, float* pair_nkl, uint8_t* consensus,
                              uint8_t* divergence, uint32_t* device_status, void* workspace,
                              size_t workspace_bytes, spec_stream_t stream);

/*
 * spec_verify_stochastic without a workspace argument: the same computation, inputs and
 * outputs, with its scratch memory inside the library. The pages have no counterpart to
 * this entry point; it exists for callers that cannot allocate device memory -- code that
 * is handed its buffers by a host framework (for example a plugin whose memory pool is
 * owned by an inference server) and must not call cudaMalloc/cudaFree, which may
 * synchronise the device or fragment a pool it does not own.
 *
 *   - Nothing is allocated: the scratch is one static device array of
 *     SPEC_STATIC_SCRATCH_BYTES bytes, present on every GPU that loads the library until
 *     the process exits. A problem whose spec_workspace_bytes(g, dtype, SPEC_MODE_STOCHASTIC)
 *     exceeds it returns SPEC_ERR_TOO_LARGE before anything runs.
 *   - The first call on each device (with that device current) looks up the array's
 *     device address with cudaGetSymbolAddress and caches it; make that first call
 *     before any stream capture. The cached address belongs to the device's primary
 *     context: after cudaDeviceReset on that device the address is stale, so do not call
 *     this entry point again in a process that has reset the device.
 *   - Every call on a device shares the one array. Calls on the same stream are ordered
 *     and safe; calls that overlap on the GPU (other streams, other host threads) race
 *     on it and give undefined results. Each call re-initialises what it needs, so no
 *     state carries over from the previous call.
 */
#define SPEC_STATIC_SCRATCH_BYTES (1u << 20)

spec_status spec_verify_stochastic_static(spec_batch g, spec_dtype dtype, const void* target_logits,
                                          const void* draft_logits, const int32_t* draft_tokens,
                                          float temperature, const float* u_accept, const float* u_sample,
                                          int32_t* n_accepted, int32_t* out_tokens, float* p_x, float* q_x,
                                          float* alpha, float* nkl, uint8_t* nkl_mask, float nkl_delta,
                                          int32_t* greedy_n, int32_t* greedy_tokens, uint32_t* device_status,
                                          spec_stream_t stream);

/* Self-test of the bounded waits (failure detection without a GPU fault): re-arms one
 * sequence in `workspace` and launches the stochastic call's sampler over it with no tile
 * kernel, so the sequence's decision is never published and the tile count never
 * completes. The sampler gives up after its poll limit (well under a second), ORs
 * SPEC_DEV_TIMEOUT into *device_status and returns; the context stays usable. Nothing is
 * read from any logits. workspace: at least spec_workspace_bytes() of a dense bf16 batch
 * with B = 1, gamma = 1, V = 8, 256-byte aligned. Host errors as for the other calls. */
spec_status spec_selftest_wait_timeout(uint32_t* device_status, void* workspace, size_t workspace_bytes,
                                       spec_stream_t stream);

/* A static English description of a spec_status value. */
const char* spec_status_str(spec_status s);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
