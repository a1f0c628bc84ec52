/*
 * kvc.h -- C ABI of libkvc: the decoding-time KV-cache eviction step on one GPU.
 *
 * The step follows the BeaconKV write-up "长推理把显存吃爆了？BeaconKV：用几个
 * 「信标查询」预判模型会回头看什么" (sections "观察 query 集 = 最近查询 + 信标查询",
 * "Continual FPS：有界内存的在线最远点采样", "打分时的 RoPE 对齐" and "实验"),
 * with per-head budgets as in the ReasonAlloc note ("Core Mechanism": a budget
 * B_{L_i,H_j} per head fed to any eviction policy).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers named in a "device" comment are CUDA device pointers (or
 *   managed memory); everything else is host memory read during the call only.
 *   The caller owns every buffer; the library allocates nothing and never
 *   synchronises the stream. Results depend only on a call's arguments. The
 *   library holds two pieces of process state, neither of which a normal call
 *   depends on: kvc_score_static's fixed device region (its scratch, see there)
 *   and the test-only switch of kvc_debug_fault (off unless a test turns it on).
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream). Every kernel is launched on it, in call order.
 * - Return value: KVC_OK (0) or a negative KVC_ERR_* code. Every argument is
 *   checked on the host BEFORE the first launch, so a call that returns an
 *   argument error has launched nothing and changed nothing.
 * - Conditions only the GPU can see (a per-head budget below prefix+recent,
 *   a query-buffer count out of range, a malformed kept-index list) are
 *   reported by OR-ing KVC_STATUS_* bits into `*status`, a caller-owned int32
 *   in device memory (may be NULL to ignore them). The affected head is left
 *   exactly as it was; the others proceed.
 * - Layout: dense, no paging. One layer of the cache is [B, Hkv, ncap, D]
 *   contiguous in the storage type; head (b, h) of layer l starts at element
 *   ((b*Hkv + h) * ncap) * D of K[l] / V[l], and its first N tokens are valid.
 *   Query head hq belongs to KV head hq / (Hq/Hkv) (contiguous groups).
 *   Per-head arrays ("[L,B,Hkv]") are flat in (l, b, h) order.
 * - Supported: storage KVC_BF16 with D in {64, 128}, KVC_F32 with D in
 *   {64, 128}; Hq % Hkv == 0; L <= KVC_MAX_LAYERS.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVC_ABI_VERSION 5
#define KVC_MAX_LAYERS 128

#if defined(__GNUC__)
#define KVC_API __attribute__((visibility("default")))
#else
#define KVC_API
#endif

typedef enum { KVC_BF16 = 0, KVC_F32 = 1 } kvc_dtype;

enum {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARG = -1,          /* null pointer, non-positive size, inconsistent sizes */
  KVC_ERR_UNSUPPORTED_DTYPE = -2,
  KVC_ERR_UNSUPPORTED_HEAD_DIM = -3, /* D not in {64, 128} */
  KVC_ERR_BUDGET_RANGE = -4,         /* uniform budget < prefix + recent */
  KVC_ERR_NOT_DIVISIBLE = -5,        /* Hq % Hkv != 0, or an odd FPS buffer size */
  KVC_ERR_LAUNCH = -6,               /* a CUDA launch or attribute call failed */
  KVC_ERR_WORKSPACE = -7,            /* workspace missing or smaller than *_workspace_size() */
  KVC_ERR_ALIGNMENT = -8,            /* a device pointer is not 16-byte aligned */
  KVC_ERR_TOO_LARGE = -9             /* a size exceeds what the kernels index with 32 bits */
};

/* Bits OR-ed into the optional device status word. */
#define KVC_STATUS_BUDGET_RANGE 0x1u /* a per-head budget < prefix + recent: head kept whole */
#define KVC_STATUS_COUNT_RANGE 0x2u  /* a query-buffer count < 0 or > qmax: head left alone */
#define KVC_STATUS_BAD_INDEX 0x4u    /* kvc_compact: kept list not strictly increasing in [k, N) */
#define KVC_STATUS_TIMEOUT 0x8u      /* a bounded device-side wait gave up; that work was skipped */

/*
 * Scoring and budget options (kvc_score, kvc_score_static, kvc_evict). A NULL
 * options pointer, or one that is all zero, selects the default step: max over
 * rows, max over the GQA group, budgets as given, no entropy output.
 *
 * Aggregation (BeaconKV write-up, "实验": the ablation of max against mean
 * aggregation of the observation queries' weights). With p_rj the softmax
 * weight of observation row r on key j, and the rows of query head g:
 *   A_g(j) = max_r p_rj             row_agg KVC_AGG_MAX
 *          = (1/M_g) sum_r p_rj     row_agg KVC_AGG_MEAN (M_g = g's valid rows)
 *   score_j = max_g A_g(j)          group_agg KVC_AGG_MAX
 *           = sum_g A_g(j)          group_agg KVC_AGG_SUM
 * Query heads without rows (no recent queries, empty buffer) take no part.
 *
 * Entropy (ReasonAlloc note, "Key Concepts": head utility from normalised
 * attention entropy): entropy[l,b,h] = mean over the KV head's valid rows of
 * H_r / ln N, H_r = -sum_j p_rj ln p_rj, in [0, 1]; 0 when N = 1.
 *
 * Head budgets (ReasonAlloc note, "Core Mechanism": budget moves from low- to
 * high-utility heads within a layer, the layer total fixed), kvc_evict only:
 * with KVC_BUDGET_ENTROPY each (layer, sequence)'s budgets are replaced by
 * kvc_head_budget's reallocation of their total by the heads' entropies.
 */
#define KVC_AGG_MAX 0
#define KVC_AGG_MEAN 1 /* row_agg only */
#define KVC_AGG_SUM 2  /* group_agg only */
#define KVC_BUDGET_GIVEN 0
#define KVC_BUDGET_ENTROPY 1
/* Scoring kernel for bf16 caches (kernel field; a test and profiling aid: every
 * kernel computes the same scores). KVC_KERNEL_AUTO picks by shape; a forced
 * kernel that does not apply to the call falls back to the automatic choice
 * (RESIDENT: 128-row tiles and short caches; SPLIT: default options only; WIDE:
 * default options and more than 128 observation rows). fp32 caches: SPLIT forces
 * the streaming passes; any other value lets a cache of at most 1024 keys per head
 * with default options take one thread-block-cluster launch after the observation
 * rows. */
#define KVC_KERNEL_AUTO 0
#define KVC_KERNEL_RESIDENT 1 /* single read of K, logits held in tensor memory */
#define KVC_KERNEL_SPLIT 2    /* two streaming passes, independent work items */
#define KVC_KERNEL_FUSED 3    /* two passes with a per-group exchange */
#define KVC_KERNEL_WIDE 4     /* two streaming passes, keys on the tensor-memory lanes (> 128 rows) */
typedef struct {
  int32_t row_agg;     /* KVC_AGG_MAX or KVC_AGG_MEAN */
  int32_t group_agg;   /* KVC_AGG_MAX or KVC_AGG_SUM */
  int32_t head_budget; /* KVC_BUDGET_GIVEN or KVC_BUDGET_ENTROPY (kvc_evict only) */
  int32_t kernel;      /* KVC_KERNEL_* (0 = automatic) */
  float* entropy;      /* [L,B,Hkv] fp32 (device, out) or NULL */
} kvc_opts;

/* One KV cache: every layer's K and V. */
typedef struct {
  int32_t dtype;   /* kvc_dtype of K and V */
  int32_t L;       /* layers */
  int32_t B;       /* sequences */
  int32_t Hq;      /* query heads per layer */
  int32_t Hkv;     /* KV heads per layer */
  int32_t D;       /* head dimension */
  int32_t N;       /* tokens currently cached in every head (== B_max at the trigger) */
  int32_t pad_;    /* must be 0 */
  int64_t ncap;    /* token capacity of every head, >= N (the head stride is ncap*D elements) */
  void* const* K;  /* host array of L device pointers, 16-byte aligned, one per layer */
  void* const* V;  /* host array of L device pointers, 16-byte aligned, one per layer */
} kvc_cache;

/*
 * kvc_fps_update -- continual farthest-point compression of the beacon buffer.
 * BeaconKV write-up, "Continual FPS：有界内存的在线最远点采样": every attention
 * head keeps a bounded buffer of pre-RoPE queries; when it reaches B_Q^max it is
 * cut back to B_Q^min by farthest-point sampling.
 *
 * For every query head whose count equals qmax: normalise the qmax buffered
 * queries, start from the oldest (row 0), repeatedly add the candidate whose
 * cosine distance 1 - cos to the chosen set is largest (ties to the lower row)
 * until qmax/2 are chosen, move the chosen rows to the buffer's front in their
 * original (time) order and set count to qmax/2. Heads with count < qmax are
 * untouched; count > qmax or < 0 sets KVC_STATUS_COUNT_RANGE and leaves the head.
 *
 *   dtype        kvc_dtype of qbuf
 *   L, B, Hq, D  sizes; qbuf is [L,B,Hq,qmax,D] (device, in/out), count is
 *                [L,B,Hq] int32 (device, in/out)
 *   qmax         buffer capacity, even, 2..64
 *   picks        [L,B,Hq,qmax/2] int32 (device, out, may be NULL): the old row
 *                index of each survivor, ascending; -1 rows for heads left alone
 *   status       device int32 or NULL
 */
KVC_API int kvc_fps_update(int32_t dtype, int32_t L, int32_t B, int32_t Hq, int32_t D, void* qbuf, int32_t qmax,
                   int32_t* count, int32_t* picks, int32_t* status, void* stream);

/*
 * kvc_append -- one decode step's queries into the observation state.
 * BeaconKV write-up, "Continual FPS：有界内存的在线最远点采样": each head's buffer of
 * pre-RoPE queries grows to B_Q^max and is cut back to B_Q^min by farthest-point
 * sampling; "观察 query 集 = 最近查询 + 信标查询": the recent observation queries are
 * the latest n_r queries at their own positions.
 *
 * For every query head, in this order:
 *   - ring: row t mod n_r of q_recent receives q_post, or, when q_post is NULL, q_pre
 *     turned to position t exactly as kvc_score turns beacons (rotate-half pairs,
 *     angle t * theta^(-2i/D) from fp64, cos/sin rounded to fp32, each product and
 *     the sum rounded to fp32, the result rounded to the storage type);
 *   - a buffer found full (count == qmax) is compressed as kvc_fps_update does
 *     (qmax/2 survivors in time order, count = qmax/2);
 *   - q_pre is written to buffer row count and count grows by one;
 *   - a buffer that has just become full is compressed the same way.
 * Rows at or past the new count are left as those writes leave them. A count < 0
 * or > qmax sets KVC_STATUS_COUNT_RANGE and leaves that head's buffer and count
 * (its ring row is still written). A decode loop calls this once per step and
 * kvc_evict (or kvc_score) with the same qbuf, count and q_recent when the cache
 * reaches B_max.
 *
 *   dtype        kvc_dtype of every query array
 *   L, B, Hq, D  sizes; query heads are flat in (l, b, hq) order
 *   q_pre        [L,B,Hq,D] this step's pre-RoPE queries (device, read)
 *   q_post       [L,B,Hq,D] this step's post-RoPE queries (device, read) or NULL
 *   t            this step's position (>= 0); rope_theta the rotary base (> 1; read
 *                only when q_post is NULL and n_r > 0)
 *   qbuf, count  [L,B,Hq,qmax,D] and [L,B,Hq] int32 (device, in/out); qmax even, 2..64
 *   q_recent     [L,B,Hq,n_r,D] ring (device, in/out); n_r in 0..64 (0: no ring, may be NULL)
 *   picks        [L,B,Hq,qmax/2] int32 (device, out) or NULL: the old rows of this
 *                call's last compression per head, ascending; -1 rows where none ran
 *   status       device int32 or NULL
 */
KVC_API int kvc_append(int32_t dtype, int32_t L, int32_t B, int32_t Hq, int32_t D, const void* q_pre,
                       const void* q_post, int64_t t, double rope_theta, void* qbuf, int32_t qmax, int32_t* count,
                       void* q_recent, int32_t n_r, int32_t* picks, int32_t* status, void* stream);

/*
 * kvc_score -- importance of every cached key from the observation queries.
 * BeaconKV write-up, "观察 query 集 = 最近查询 + 信标查询" and "打分时的 RoPE 对齐":
 * the observation set is the recent queries at their own positions plus beacon
 * queries rotated to the current step t; a key's importance is the max over the
 * observation set of its attention weight, so one beacon that cares is enough.
 *
 * Per KV head (l, b, h), the observation rows are, for each of its G = Hq/Hkv
 * query heads: the n_r recent queries as given (post-RoPE), then its beacons.
 * The beacons are the buffer's first count rows when count <= n_b, else the
 * farthest-point choice of n_b of them (as kvc_fps_update, buffer unchanged),
 * each rotated to position t (rotate-half pairs (i, i+D/2), angle
 * t * theta^(-2i/D), cos/sin in fp64) and rounded to the storage type. Then
 *     scores[j] = max over rows r of exp(s_rj - lse_r),  s_rj = q_r . k_j / sqrt(D),
 *     lse_r = log sum_{j<N} exp(s_rj),
 * over all N cached keys, in fp32 with fp32 accumulation.
 *
 *   c            the cache (K read only; V unused)
 *   q_recent     [L,B,Hq,n_r,D] storage type (device), n_r in 0..64
 *   qbuf, count  as kvc_fps_update (device, read only); qmax in 0..64
 *   n_b          beacons per query head, 0..qmax; n_r + n_b >= 1
 *   t, rope_theta  current step and rotary base (theta > 1)
 *   scores       [L,B,Hkv,N] fp32 (device, out)
 *   beacon_picks [L,B,Hq,n_b] int32 (device, out, may be NULL): buffer rows used
 *                as beacons, ascending, -1 padded
 *   opts         NULL or the aggregation variant / entropy output (see kvc_opts;
 *                head_budget must be KVC_BUDGET_GIVEN here). A variant other than
 *                max/max, or an entropy output, stores each query head's rows from
 *                a 16-row boundary; G * that stride must stay within 256 rows
 *                (else KVC_ERR_TOO_LARGE).
 *   workspace    device scratch of at least kvc_score_workspace_size() bytes,
 *                256-byte aligned; contents on entry do not matter
 */
KVC_API size_t kvc_score_workspace_size(const kvc_cache* c, int32_t n_r, int32_t n_b);
KVC_API int kvc_score(const kvc_cache* c, const void* q_recent, int32_t n_r, const void* qbuf, const int32_t* count,
              int32_t qmax, int32_t n_b, int64_t t, double rope_theta, float* scores, int32_t* beacon_picks,
              const kvc_opts* opts, void* workspace, size_t ws_bytes, void* stream);

/*
 * kvc_select -- which tokens each head keeps.
 * BeaconKV write-up, end of "打分时的 RoPE 对齐": prefix tokens and the most
 * recent tokens are always kept and the rest of the budget is filled by top
 * score; "实验": on reaching B_KV^max the cache drops to 7/8 B_KV^max. ReasonAlloc
 * note, "Core Mechanism": the budget may differ per head.
 *
 * Per head with budget b (the head's total kept count): if b >= N keep all;
 * else keep [0, prefix), [N-recent, N) and the b - prefix - recent highest
 * scores of [prefix, N-recent), equal scores going to the lower index.
 * kept_idx receives the kept token indices in ascending order.
 *
 *   scores       [L,B,Hkv,N] fp32 (device); ranked by value (any finite value, -0 equal
 *                to +0; a NaN with the sign bit clear ranks above +inf, one with it set
 *                below -inf)
 *   budget       [L,B,Hkv] int32 (device) or NULL to use budget_all for all heads;
 *                an entry < prefix + recent sets KVC_STATUS_BUDGET_RANGE and
 *                keeps that head whole
 *   kept_idx     [L,B,Hkv,N] int32 (device, out); entries past kept_len are not written
 *   kept_len     [L,B,Hkv] int32 (device, out)
 */
KVC_API int kvc_select(const float* scores, int32_t L, int32_t B, int32_t Hkv, int32_t N, int32_t prefix, int32_t recent,
               const int32_t* budget, int32_t budget_all, int32_t* kept_idx, int32_t* kept_len, int32_t* status,
               void* stream);

/*
 * kvc_compact -- move the kept tokens' K and V rows to the head's front, in
 * their original order, in place. The kept tokens of the BeaconKV write-up's
 * policy stay; evicted slots are reused. Rows past kept_len keep their old bytes.
 *
 *   kept_idx, kept_len   as produced by kvc_select (device). Each head's list is
 *                checked first (strictly increasing, kept_idx[k] in [k, N),
 *                kept_len <= N); a bad list sets KVC_STATUS_BAD_INDEX and that
 *                head is not touched.
 * The caller then treats head h's length as kept_len[h].
 */
KVC_API int kvc_compact(const kvc_cache* c, const int32_t* kept_idx, const int32_t* kept_len, int32_t* status,
                void* stream);

/*
 * kvc_evict -- the whole eviction step: beacons, scores, selection and
 * compaction for every (l, b, h) of the cache, on one stream. Equivalent to
 * kvc_score, kvc_select and kvc_compact in sequence (same arguments); the
 * intermediate arrays live in the workspace unless the caller asks for them.
 *
 *   scores       [L,B,Hkv,N] fp32 (device, out) or NULL
 *   kept_idx     [L,B,Hkv,N] int32 (device, out) or NULL
 *   kept_len     [L,B,Hkv] int32 (device, out), required
 *   opts         NULL or options (see kvc_opts); with KVC_BUDGET_ENTROPY the budgets
 *                (budget or budget_all) are each layer's preallocation, reallocated
 *                over its heads as kvc_head_budget does before selection
 *   workspace    at least kvc_evict_workspace_size() bytes, 256-byte aligned
 */
KVC_API size_t kvc_evict_workspace_size(const kvc_cache* c, int32_t n_r, int32_t n_b);
KVC_API int kvc_evict(const kvc_cache* c, const void* q_recent, int32_t n_r, const void* qbuf, const int32_t* count,
              int32_t qmax, int32_t n_b, int64_t t, double rope_theta, int32_t prefix, int32_t recent,
              const int32_t* budget, int32_t budget_all, int32_t* kept_idx, int32_t* kept_len, float* scores,
              int32_t* status, const kvc_opts* opts, void* workspace, size_t ws_bytes, void* stream);

/*
 * kvc_score_static -- kvc_score for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a deployment convenience of this library.
 *
 * Some callers cannot call cudaMalloc or hand the library a workspace: a serving
 * runtime that reserves all device memory up front for weights and its KV pool, or
 * code that runs where allocation is not allowed (inside an allocator callback or an
 * out-of-memory recovery path). This entry point computes exactly what kvc_score
 * computes (same arguments, same results) but takes its scratch from a fixed region
 * of KVC_STATIC_SCRATCH_BYTES that the library reserves in device memory when it is
 * loaded; every GPU that loads the library holds that region until the process exits.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * - Size limit: the call is rejected with KVC_ERR_WORKSPACE, before any launch, when
 *   kvc_score_workspace_size() for these arguments exceeds KVC_STATIC_SCRATCH_BYTES
 *   (the Qwen3-4B-shaped step, about 11.9 MB, fits; larger caches do not).
 * - Set-up: every call looks up the region's device address in the calling thread's
 *   current context (cudaGetSymbolAddress, with the device current), so a context that
 *   was reset and made again gets its own region. The first call on a device also loads
 *   the library's device code there: make that first call before any CUDA stream capture.
 * - Sharing: every call on a device uses the same region and leaves its contents behind
 *   (the library clears what must start at zero). Calls whose kernels overlap on the GPU
 *   (two streams, or two threads) race on the region: order them on one stream.
 */
#define KVC_STATIC_SCRATCH_BYTES (16u << 20)
KVC_API int kvc_score_static(const kvc_cache* c, const void* q_recent, int32_t n_r, const void* qbuf,
                             const int32_t* count, int32_t qmax, int32_t n_b, int64_t t, double rope_theta,
                             float* scores, int32_t* beacon_picks, const kvc_opts* opts, void* stream);

/*
 * kvc_head_budget -- online head-wise budgets from attention entropy.
 * ReasonAlloc note, "Core Mechanism": each layer's preallocated budget is moved
 * from low-utility to high-utility heads, the layer total held fixed; "Key
 * Concepts": utility from normalised attention entropy, low entropy gets more.
 * The note states no formula; per (layer, sequence) with H = Hkv heads:
 *   T = sum_h min(given_h, N); f = prefix + recent; cap = N - f;
 *   u_h = 1 - entropy_h clipped to [0, 1];
 *   the E = T - H f slots above the floors are shared in proportion to u
 *   (equally if every remaining u is 0); a share above cap is cut to cap and
 *   the rest shared again among the other heads (water-filling);
 *   integer shares by largest remainder, ties to the lower head;
 *   budget_out_h = f + share_h.
 * fp64, every operation rounded on its own, heads in order. If N <= f or
 * T >= H N, budget_out_h = min(given_h, N). A given_h < f sets
 * KVC_STATUS_BUDGET_RANGE and that (layer, sequence) keeps its given budgets.
 *
 *   entropy      [L,B,Hkv] fp32 (device), e.g. kvc_opts.entropy of kvc_score
 *   budget       [L,B,Hkv] int32 (device) or NULL to use budget_all for all heads
 *   budget_out   [L,B,Hkv] int32 (device, out); may alias budget
 *   status       device int32 or NULL
 */
KVC_API int kvc_head_budget(const float* entropy, int32_t L, int32_t B, int32_t Hkv, int32_t N, int32_t prefix,
                            int32_t recent, const int32_t* budget, int32_t budget_all, int32_t* budget_out,
                            int32_t* status, void* stream);

/*
 * kvc_epikv_score -- the EPIKV eviction score from two layers' hidden states.
 * EPIKV write-up, "方法论：EPIKV": a token's signal at layer l is how far the
 * residual stream moves when it is decoded, g_l(t) = ||h_l(t) - h_l(t-1)||_2;
 * it is corrected for position by a causal rolling z-score
 * z_l(t) = (g_l(t) - mu_l(t)) / (sigma_l(t) + eps), and the eviction score is
 * z_A(t) - z_B(t) for a layer of the band where change marks important tokens (A)
 * and one where it marks predictable ones (B). Higher scores are kept. The
 * write-up states no window, eps or first-token rule; here g(0) = 0, token 0 lies
 * in no window, window(t) = tokens max(1, t-W+1)..t, sigma is the population
 * deviation; g in fp32, the window's mean and variance in fp64 (prefix sums), sigma and
 * the quotient in fp32.
 *
 *   dtype        kvc_dtype of hA, hB
 *   B, N, dm     sequences, tokens, hidden size; dm a multiple of 8 (bf16) or 4
 *                (fp32), at most 8192 (bf16) or 4096 (fp32)
 *   hA, hB       [B,N,dm] hidden states of layers A and B (device, 16-byte aligned)
 *   window, eps  W >= 1 tokens; eps > 0 (a constant window has sigma 0)
 *   g            [2,B,N] fp32 (device, out) or NULL: g_A then g_B
 *   scores       [B,N] fp32 (device, out)
 *   workspace    at least kvc_epikv_workspace_size(B, N) bytes, 256-byte aligned
 */
KVC_API size_t kvc_epikv_workspace_size(int32_t B, int32_t N);
KVC_API int kvc_epikv_score(int32_t dtype, int32_t B, int32_t N, int32_t dm, const void* hA, const void* hB,
                            int32_t window, float eps, float* g, float* scores, void* workspace, size_t ws_bytes,
                            void* stream);

/*
 * kvc_epikv_evict -- eviction by the EPIKV score: kvc_epikv_score over the cache's
 * B sequences and N tokens, then one selection per sequence (kvc_select's rule:
 * [0, prefix) and [N-recent, N) kept, the rest of the budget by highest score,
 * ties to the lower index) whose kept list compacts every layer and KV head of that
 * sequence in place (kvc_compact's move). The score is a property of the token,
 * so all heads of a sequence keep the same tokens.
 *
 *   c            the cache (K and V moved); its dtype is the hidden states' type
 *   hA, hB, dm, window, eps   as kvc_epikv_score
 *   budget       [B] int32 kept total per sequence (device) or NULL for budget_all
 *   kept_idx     [B,N] int32 (device, out) or NULL; kept_len [B] int32 (device, out)
 *   scores       [B,N] fp32 (device, out) or NULL
 *   workspace    at least kvc_epikv_workspace_size(B, N) bytes, 256-byte aligned
 */
KVC_API int kvc_epikv_evict(const kvc_cache* c, const void* hA, const void* hB, int32_t dm, int32_t window, float eps,
                            int32_t prefix, int32_t recent, const int32_t* budget, int32_t budget_all,
                            int32_t* kept_idx, int32_t* kept_len, float* scores, int32_t* status, void* workspace,
                            size_t ws_bytes, void* stream);

/* Number of kernels one kvc_evict call with these arguments and default options
 * launches (host only; for accounting, e.g. counting launches inside a timed region;
 * it queries the current device's SM count and shared memory). 0 for a bad cache. */
KVC_API int kvc_evict_launch_count(const kvc_cache* c, int32_t n_r, int32_t n_b);

/* Human-readable text for a KVC_ERR_* code (static storage). */
KVC_API const char* kvc_strerror(int code);

/* KVC_ABI_VERSION of the loaded library. */
KVC_API int kvc_abi_version(void);

/* Test-only fault switch for the failure-detection path; none of the pages has a counterpart.
 * mode 1: from the next scoring launch on, the first CTA of the single-read scoring kernel
 * (bf16 caches with 128-row observation tiles) withholds its exchange partials, so its group's
 * bounded waits give up after about 50 ms: those heads' scores are left unset,
 * KVC_STATUS_TIMEOUT is raised in the status word of kvc_evict, and the launch still returns.
 * mode 0 restores normal behaviour. Process-wide, not thread-safe against concurrent calls.
 * Returns KVC_OK or KVC_ERR_INVALID_ARG for any other mode. */
KVC_API int kvc_debug_fault(int32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H_ */
