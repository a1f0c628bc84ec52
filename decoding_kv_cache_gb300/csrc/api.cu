// api.cu -- the extern "C" entry points of libkvc: argument checks, workspace layout, launches.
//
// Every check happens on the host before the first launch of a call, so a rejected call
// has touched nothing. Conditions that only the device can see are OR-ed into the
// caller's status word by the kernels (see kvc.h).
#include <atomic>
#include <math.h>
#include <string.h>

#include "kvc_internal.cuh"

namespace kvc {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dtype_dim(int dtype, int D) {
  if (dtype != KVC_BF16 && dtype != KVC_F32) return KVC_ERR_UNSUPPORTED_DTYPE;
  if (D != 64 && D != 128) return KVC_ERR_UNSUPPORTED_HEAD_DIM;
  return KVC_OK;
}

// Validates the cache description and copies its layer pointers.
int check_cache(const kvc_cache* c, CacheGeom* g, LayerPtrs* K, LayerPtrs* V) {
  if (!c || !c->K || !c->V) return KVC_ERR_INVALID_ARG;
  int rc = check_dtype_dim(c->dtype, c->D);
  if (rc) return rc;
  if (c->L < 1 || c->L > KVC_MAX_LAYERS || c->B < 1 || c->Hq < 1 || c->Hkv < 1 || c->N < 1 || c->pad_ != 0)
    return KVC_ERR_INVALID_ARG;
  if (c->Hq % c->Hkv) return KVC_ERR_NOT_DIVISIBLE;
  if (c->ncap < c->N) return KVC_ERR_INVALID_ARG;
  const long long heads = (long long)c->L * c->B * c->Hkv;
  if (heads > 65535 || (long long)c->N > (1LL << 30) || (long long)c->B * c->Hq * c->L > (1LL << 30))
    return KVC_ERR_TOO_LARGE;
  for (int l = 0; l < c->L; ++l) {
    if (!c->K[l] || !c->V[l]) return KVC_ERR_INVALID_ARG;
    if (!aligned16(c->K[l]) || !aligned16(c->V[l])) return KVC_ERR_ALIGNMENT;
    K->p[l] = c->K[l];
    V->p[l] = c->V[l];
  }
  for (int l = c->L; l < KVC_MAX_LAYERS; ++l) K->p[l] = V->p[l] = nullptr;
  *g = CacheGeom{c->L, c->B, c->Hq, c->Hkv, c->D, c->N, (long long)c->ncap};
  return KVC_OK;
}

// The options of one call, checked; ext = the extended scoring epilogue is needed.
struct Opts {
  bool ext;
  int row_agg, group_agg, head_budget;
  int kernel;      // KVC_KERNEL_* (a test and profiling aid)
  float* entropy;  // the caller's entropy output, or null
};

int check_opts(const kvc_opts* o, bool evict, Opts* out) {
  *out = Opts{false, KVC_AGG_MAX, KVC_AGG_MAX, KVC_BUDGET_GIVEN, KVC_KERNEL_AUTO, nullptr};
  if (!o) return KVC_OK;
  if ((o->row_agg != KVC_AGG_MAX && o->row_agg != KVC_AGG_MEAN) ||
      (o->group_agg != KVC_AGG_MAX && o->group_agg != KVC_AGG_SUM) ||
      (o->head_budget != KVC_BUDGET_GIVEN && o->head_budget != KVC_BUDGET_ENTROPY) || o->kernel < KVC_KERNEL_AUTO ||
      o->kernel > KVC_KERNEL_WIDE)
    return KVC_ERR_INVALID_ARG;
  if (!evict && o->head_budget != KVC_BUDGET_GIVEN) return KVC_ERR_INVALID_ARG;
  if (o->entropy && (reinterpret_cast<uintptr_t>(o->entropy) & 3u)) return KVC_ERR_ALIGNMENT;
  out->row_agg = o->row_agg;
  out->group_agg = o->group_agg;
  out->head_budget = o->head_budget;
  out->kernel = o->kernel;
  out->entropy = o->entropy;
  out->ext = o->row_agg != KVC_AGG_MAX || o->group_agg != KVC_AGG_MAX || o->entropy ||
             o->head_budget == KVC_BUDGET_ENTROPY;
  return KVC_OK;
}

int check_queries(const kvc_cache* c, const void* q_recent, int n_r, const void* qbuf, const int32_t* count,
                  int qmax, int n_b, double theta, bool ext) {
  if (n_r < 0 || n_r > 64 || qmax < 0 || qmax > kMaxQmax || n_b < 0 || n_b > qmax || n_r + n_b < 1)
    return KVC_ERR_INVALID_ARG;
  if (n_r > 0 && !q_recent) return KVC_ERR_INVALID_ARG;
  if (qmax > 0 && (!qbuf || !count)) return KVC_ERR_INVALID_ARG;
  if (!(theta > 1.0) || !isfinite(theta)) return KVC_ERR_INVALID_ARG;
  const int G = c->Hq / c->Hkv;
  if ((long long)(G - 1) * obs_qstride(n_r, n_b, ext) + n_r + n_b > kMaxRows) return KVC_ERR_TOO_LARGE;
  if ((q_recent && !aligned16(q_recent)) || (qbuf && !aligned16(qbuf))) return KVC_ERR_ALIGNMENT;
  return KVC_OK;
}

namespace {
std::atomic<int> g_debug_fault{0};  // test-only fault switch, read at each scoring launch
}

// Rotary angles of step t in fp64 (BeaconKV write-up, "打分时的 RoPE 对齐": beacons are turned
// to position t): pair (i, i + D/2) turns by t * theta^(-2i/D); cos and sin rounded to fp32.
void rope_table(float2 (&rope)[64], int D, int64_t t, double theta) {
  for (int i = 0; i < D / 2; ++i) {
    const double ang = (double)t * pow(theta, -2.0 * (double)i / (double)D);
    rope[i] = make_float2((float)cos(ang), (float)sin(ang));
  }
  for (int i = D / 2; i < 64; ++i) rope[i] = make_float2(0.f, 0.f);
}

void fill_score_args(ScoreArgs* a, const CacheGeom& g, int dtype, const LayerPtrs& K, const void* q_recent, int n_r,
                     const void* qbuf, const int32_t* count, int qmax, int n_b, int64_t t, double theta,
                     float* scores, int32_t* beacon_picks, int32_t* status, const Opts& o, float* entropy) {
  memset(a, 0, sizeof(*a));  // every field starts defined (no exchange words to zero, one tile)
  a->g = g;
  a->ext = o.ext ? 1 : 0;
  a->qstride = obs_qstride(n_r, n_b, o.ext);
  a->row_agg = o.row_agg;
  a->group_agg = o.group_agg;
  a->entropy = entropy;
  a->tiles = 1;  // launch_score may split 256-row tiles
  a->kernel = o.kernel;
  a->debug_fault = g_debug_fault.load();
  a->dtype = dtype;
  a->K = K;
  a->q_recent = q_recent;
  a->n_r = n_r;
  a->qbuf = qbuf;
  a->count = count;
  a->qmax = qmax;
  a->n_b = n_b;
  a->t = (long long)t;
  a->theta = theta;
  a->scores = scores;
  a->beacon_picks = beacon_picks;
  a->status = status;
  a->M = obs_rows_used(g.Hq / g.Hkv, n_r, n_b, o.ext);
  a->M_pad = obs_rows(a->M, dtype);
  a->M_n = (a->M + 15) / 16 * 16;
  rope_table(a->rope, g.D, t, theta);
  a->nchunk = (g.N + kChunk - 1) / kChunk;
}

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace
}  // namespace kvc

using namespace kvc;

extern "C" {

int kvc_abi_version(void) { return KVC_ABI_VERSION; }

int kvc_debug_fault(int32_t mode) {
  if (mode < 0 || mode > 1) return KVC_ERR_INVALID_ARG;
  g_debug_fault.store(mode);
  return KVC_OK;
}

int kvc_head_budget(const float* entropy, int32_t L, int32_t B, int32_t Hkv, int32_t N, int32_t prefix,
                    int32_t recent, const int32_t* budget, int32_t budget_all, int32_t* budget_out, int32_t* status,
                    void* stream) {
  if (!entropy || !budget_out || L < 1 || B < 1 || Hkv < 1 || N < 1 || prefix < 0 || recent < 0)
    return KVC_ERR_INVALID_ARG;
  if (Hkv > 64) return KVC_ERR_TOO_LARGE;
  const long long groups = (long long)L * B;
  if (groups > (1LL << 31) - 1) return KVC_ERR_TOO_LARGE;
  if (!budget && budget_all < prefix + recent && budget_all < N) return KVC_ERR_BUDGET_RANGE;
  return launch_head_budget(entropy, (int)groups, Hkv, N, prefix, recent, budget, budget_all, budget_out, status,
                            static_cast<cudaStream_t>(stream));
}

int kvc_evict_launch_count(const kvc_cache* c, int32_t n_r, int32_t n_b) {
  CacheGeom g;
  LayerPtrs K, V;
  if (!c || n_r < 0 || n_b < 0) return 0;
  kvc_cache probe = *c;
  if (check_cache(&probe, &g, &K, &V)) return 0;
  // + selection and compaction: none for the fp32 cluster kernel (they run in it), one launch up to
  // kSelectCompactMaxN tokens per head, else two
  if (evict_fused_small(g, c->dtype, n_r, n_b)) return score_launches(g, c->dtype, n_r, n_b, false);
  return score_launches(g, c->dtype, n_r, n_b, false) + (g.N <= kSelectCompactMaxN ? 1 : 2);
}

const char* kvc_strerror(int code) {
  switch (code) {
    case KVC_OK: return "ok";
    case KVC_ERR_INVALID_ARG: return "invalid argument";
    case KVC_ERR_UNSUPPORTED_DTYPE: return "unsupported storage type";
    case KVC_ERR_UNSUPPORTED_HEAD_DIM: return "unsupported head dimension (64 or 128)";
    case KVC_ERR_BUDGET_RANGE: return "budget smaller than prefix + recent";
    case KVC_ERR_NOT_DIVISIBLE: return "query heads not a multiple of KV heads, or odd buffer size";
    case KVC_ERR_LAUNCH: return "CUDA launch failed";
    case KVC_ERR_WORKSPACE: return "workspace missing or too small";
    case KVC_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
    case KVC_ERR_TOO_LARGE: return "size too large";
    default: return "unknown error";
  }
}

int kvc_fps_update(int32_t dtype, int32_t L, int32_t B, int32_t Hq, int32_t D, void* qbuf, int32_t qmax,
                   int32_t* count, int32_t* picks, int32_t* status, void* stream) {
  int rc = check_dtype_dim(dtype, D);
  if (rc) return rc;
  if (L < 1 || B < 1 || Hq < 1 || !qbuf || !count || qmax < 2 || qmax > kMaxQmax) return KVC_ERR_INVALID_ARG;
  if (qmax % 2) return KVC_ERR_NOT_DIVISIBLE;
  const long long nq = (long long)L * B * Hq;
  if (nq > (1LL << 30)) return KVC_ERR_TOO_LARGE;
  if (!aligned16(qbuf)) return KVC_ERR_ALIGNMENT;
  return launch_fps_update(dtype, (int)nq, D, qbuf, qmax, count, picks, status, static_cast<cudaStream_t>(stream));
}

int kvc_append(int32_t dtype, int32_t L, int32_t B, int32_t Hq, int32_t D, const void* q_pre, const void* q_post,
               int64_t t, double rope_theta, void* qbuf, int32_t qmax, int32_t* count, void* q_recent, int32_t n_r,
               int32_t* picks, int32_t* status, void* stream) {
  int rc = check_dtype_dim(dtype, D);
  if (rc) return rc;
  if (L < 1 || B < 1 || Hq < 1 || !q_pre || !qbuf || !count || qmax < 2 || qmax > kMaxQmax || n_r < 0 ||
      n_r > 64 || t < 0)
    return KVC_ERR_INVALID_ARG;
  if (qmax % 2) return KVC_ERR_NOT_DIVISIBLE;
  if (n_r > 0 && !q_recent) return KVC_ERR_INVALID_ARG;
  if (n_r > 0 && !q_post && (!(rope_theta > 1.0) || !isfinite(rope_theta))) return KVC_ERR_INVALID_ARG;
  const long long nq = (long long)L * B * Hq;
  if (nq > (1LL << 30)) return KVC_ERR_TOO_LARGE;
  if (!aligned16(q_pre) || !aligned16(qbuf) || (q_post && !aligned16(q_post)) || (q_recent && !aligned16(q_recent)))
    return KVC_ERR_ALIGNMENT;
  AppendArgs a;
  a.q_pre = q_pre;
  a.q_post = q_post;
  a.qbuf = qbuf;
  a.count = count;
  a.q_recent = n_r > 0 ? q_recent : nullptr;
  a.picks = picks;
  a.status = status;
  a.nheads = (int)nq;
  a.qmax = qmax;
  a.n_r = n_r;
  a.ring_slot = n_r > 0 ? (int)(t % n_r) : 0;
  if (n_r > 0 && !q_post)
    rope_table(a.rope, D, t, rope_theta);
  else
    for (int i = 0; i < 64; ++i) a.rope[i] = make_float2(0.f, 0.f);
  return launch_append(a, dtype, D, static_cast<cudaStream_t>(stream));
}

size_t kvc_score_workspace_size(const kvc_cache* c, int32_t n_r, int32_t n_b) {
  CacheGeom g;
  LayerPtrs K, V;
  if (!c || n_r < 0 || n_b < 0) return 0;
  kvc_cache probe = *c;
  if (check_cache(&probe, &g, &K, &V)) return 0;
  // enough for either row layout (the extended one may need more rows)
  const size_t a = score_ws_bytes(g, c->dtype, n_r, n_b, false, nullptr, nullptr);
  const size_t b = score_ws_bytes(g, c->dtype, n_r, n_b, true, nullptr, nullptr);
  return a > b ? a : b;
}

int kvc_score(const kvc_cache* c, const void* q_recent, int32_t n_r, const void* qbuf, const int32_t* count,
              int32_t qmax, int32_t n_b, int64_t t, double rope_theta, float* scores, int32_t* beacon_picks,
              const kvc_opts* opts, void* workspace, size_t ws_bytes, void* stream) {
  CacheGeom g;
  LayerPtrs K, V;
  Opts o;
  int rc = check_cache(c, &g, &K, &V);
  if (rc) return rc;
  rc = check_opts(opts, false, &o);
  if (rc) return rc;
  rc = check_queries(c, q_recent, n_r, qbuf, count, qmax, n_b, rope_theta, o.ext);
  if (rc) return rc;
  if (!scores) return KVC_ERR_INVALID_ARG;
  const size_t need = score_ws_bytes(g, c->dtype, n_r, n_b, o.ext, nullptr, nullptr);
  if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return KVC_ERR_WORKSPACE;
  ScoreWs ws;
  score_ws_bytes(g, c->dtype, n_r, n_b, o.ext, &ws, workspace);
  ScoreArgs a;
  fill_score_args(&a, g, c->dtype, K, q_recent, n_r, qbuf, count, qmax, n_b, t, rope_theta, scores, beacon_picks,
                  nullptr, o, o.entropy);
  return launch_score(a, ws, static_cast<cudaStream_t>(stream));
}

int kvc_select(const float* scores, int32_t L, int32_t B, int32_t Hkv, int32_t N, int32_t prefix, int32_t recent,
               const int32_t* budget, int32_t budget_all, int32_t* kept_idx, int32_t* kept_len, int32_t* status,
               void* stream) {
  if (!scores || !kept_idx || !kept_len || L < 1 || B < 1 || Hkv < 1 || N < 1 || prefix < 0 || recent < 0)
    return KVC_ERR_INVALID_ARG;
  const long long heads = (long long)L * B * Hkv;
  if (heads > (1LL << 31) - 1 || (long long)N > (1LL << 30)) return KVC_ERR_TOO_LARGE;
  if (!budget && budget_all < prefix + recent && budget_all < N) return KVC_ERR_BUDGET_RANGE;
  return launch_select(scores, (int)heads, N, prefix, recent, budget, budget_all, nullptr, 1, kept_idx, kept_len,
                       status, static_cast<cudaStream_t>(stream));
}

int kvc_compact(const kvc_cache* c, const int32_t* kept_idx, const int32_t* kept_len, int32_t* status,
                void* stream) {
  CacheGeom g;
  LayerPtrs K, V;
  int rc = check_cache(c, &g, &K, &V);
  if (rc) return rc;
  if (!kept_idx || !kept_len) return KVC_ERR_INVALID_ARG;
  return launch_compact(g, c->dtype, K, V, kept_idx, kept_len, status, true, static_cast<cudaStream_t>(stream));
}

size_t kvc_evict_workspace_size(const kvc_cache* c, int32_t n_r, int32_t n_b) {
  const size_t sw = kvc_score_workspace_size(c, n_r, n_b);
  if (!sw) return 0;
  const size_t heads = (size_t)c->L * c->B * c->Hkv;
  const size_t per = heads * (size_t)c->N * 4;
  // scores and kept indices (used when the caller passes NULL), and the heads' order for the
  // selection and compaction
  return sw + 2 * align256(per) + align256(heads * 4);
}

int kvc_evict(const kvc_cache* c, const void* q_recent, int32_t n_r, const void* qbuf, const int32_t* count,
              int32_t qmax, int32_t n_b, int64_t t, double rope_theta, int32_t prefix, int32_t recent,
              const int32_t* budget, int32_t budget_all, int32_t* kept_idx, int32_t* kept_len, float* scores,
              int32_t* status, const kvc_opts* opts, void* workspace, size_t ws_bytes, void* stream) {
  CacheGeom g;
  LayerPtrs K, V;
  Opts o;
  int rc = check_cache(c, &g, &K, &V);
  if (rc) return rc;
  rc = check_opts(opts, true, &o);
  if (rc) return rc;
  rc = check_queries(c, q_recent, n_r, qbuf, count, qmax, n_b, rope_theta, o.ext);
  if (rc) return rc;
  if (!kept_len || prefix < 0 || recent < 0) return KVC_ERR_INVALID_ARG;
  if (!budget && budget_all < prefix + recent && budget_all < c->N) return KVC_ERR_BUDGET_RANGE;
  if (o.head_budget == KVC_BUDGET_ENTROPY && g.Hkv > 64) return KVC_ERR_TOO_LARGE;
  const size_t sw = score_ws_bytes(g, c->dtype, n_r, n_b, o.ext, nullptr, nullptr);
  const size_t per = align256((size_t)g.L * g.B * g.Hkv * (size_t)g.N * 4);
  const size_t ord = align256((size_t)g.L * g.B * g.Hkv * 4);
  if (!workspace || ws_bytes < sw + 2 * per + ord || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return KVC_ERR_WORKSPACE;
  char* wb = static_cast<char*>(workspace);
  ScoreWs ws;
  score_ws_bytes(g, c->dtype, n_r, n_b, o.ext, &ws, wb);
  float* sc = scores ? scores : reinterpret_cast<float*>(wb + sw);
  int32_t* ki = kept_idx ? kept_idx : reinterpret_cast<int32_t*>(wb + sw + per);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the entropy goes to the caller's array, else (when the budgets need it) to the workspace's
  float* ent = o.entropy ? o.entropy : (o.head_budget == KVC_BUDGET_ENTROPY ? ws.ent : nullptr);
  ScoreArgs a;
  fill_score_args(&a, g, c->dtype, K, q_recent, n_r, qbuf, count, qmax, n_b, t, rope_theta, sc, nullptr, status, o,
                  ent);
  const float* sel_ent = o.head_budget == KVC_BUDGET_ENTROPY ? ent : nullptr;
  // per-head budgets as given: the selection-and-compaction CTAs take the heads largest budget first
  // (the order is written by the observation kernel, which every path to that kernel runs first)
  int32_t* order = nullptr;
  if (budget && !sel_ent && g.N <= kSelectCompactMaxN) {
    order = reinterpret_cast<int32_t*>(wb + sw + 2 * per);
    a.order_budget = budget;
    a.order = order;
  }
  // fp32 caches of at most 1024 tokens per head: scoring, selection and compaction in one cluster launch
  SmallEvict ev;
  memset(&ev, 0, sizeof(ev));
  ev.V = V;
  ev.P = prefix;
  ev.R = recent;
  ev.budget_all = budget_all;
  ev.budget = budget;
  ev.kept_idx = ki;
  ev.kept_len = kept_len;
  bool fused = false;
  rc = launch_score(a, ws, s, sel_ent ? nullptr : &ev, &fused);
  if (rc || fused) return rc;
  if (g.N <= kSelectCompactMaxN)  // one CTA per head selects, then moves the head's K and V
    return launch_select_compact(order, sc, g, c->dtype, K, V, prefix, recent, budget, budget_all, sel_ent, ki, kept_len,
                                 status, s);
  rc = launch_select(sc, g.L * g.B * g.Hkv, g.N, prefix, recent, budget, budget_all, sel_ent, g.Hkv, ki, kept_len,
                     status, s);
  if (rc) return rc;
  return launch_compact(g, c->dtype, K, V, ki, kept_len, status, false, s);
}

// ---------------------------------------------------------------------------
// EPIKV: hidden-state scores, one kept list per sequence.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace kvc {
namespace {
struct EpikvWs {
  float* g;
  double* pre;
  uint32_t* keys;
  float* scores;
  int32_t* kept;
};
// layout: g [2][B][N] fp32, pre [2][2][B][N+1] fp64, keys [B][N], scores [B][N], kept [B][N]
size_t epikv_ws(int B, int N, EpikvWs* w, void* base) {
  const size_t bn = (size_t)B * N;
  size_t off = 0;
  const size_t o_g = off;     off += align256(2 * bn * sizeof(float));
  const size_t o_pre = off;   off += align256(4 * (size_t)B * (N + 1) * sizeof(double));
  const size_t o_keys = off;  off += align256(bn * sizeof(uint32_t));
  const size_t o_sc = off;    off += align256(bn * sizeof(float));
  const size_t o_kept = off;  off += align256(bn * sizeof(int32_t));
  if (w) {
    char* b = static_cast<char*>(base);
    w->g = reinterpret_cast<float*>(b + o_g);
    w->pre = reinterpret_cast<double*>(b + o_pre);
    w->keys = reinterpret_cast<uint32_t*>(b + o_keys);
    w->scores = reinterpret_cast<float*>(b + o_sc);
    w->kept = reinterpret_cast<int32_t*>(b + o_kept);
  }
  return off;
}
int check_epikv(int dtype, int B, int N, int dm, const void* hA, const void* hB, int W, float eps) {
  if (dtype != KVC_BF16 && dtype != KVC_F32) return KVC_ERR_UNSUPPORTED_DTYPE;
  if (B < 1 || N < 1 || dm < 1 || !hA || !hB || W < 1 || !(eps > 0.f) || !isfinite(eps)) return KVC_ERR_INVALID_ARG;
  const int per = dtype == KVC_BF16 ? 8 : 4;
  if (dm % per || dm / per > 4 * 256) return KVC_ERR_UNSUPPORTED_HEAD_DIM;
  if ((long long)B > 65535 || (long long)N > (1LL << 30) || (long long)B * N * dm > (1LL << 40)) return KVC_ERR_TOO_LARGE;
  if (!aligned16(hA) || !aligned16(hB)) return KVC_ERR_ALIGNMENT;
  return KVC_OK;
}
}  // namespace
}  // namespace kvc

extern "C" {

size_t kvc_epikv_workspace_size(int32_t B, int32_t N) {
  if (B < 1 || N < 1) return 0;
  return epikv_ws(B, N, nullptr, nullptr);
}

int kvc_epikv_score(int32_t dtype, int32_t B, int32_t N, int32_t dm, const void* hA, const void* hB, int32_t window,
                    float eps, float* g, float* scores, void* workspace, size_t ws_bytes, void* stream) {
  int rc = check_epikv(dtype, B, N, dm, hA, hB, window, eps);
  if (rc) return rc;
  if (!scores) return KVC_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < epikv_ws(B, N, nullptr, nullptr) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return KVC_ERR_WORKSPACE;
  EpikvWs w;
  epikv_ws(B, N, &w, workspace);
  return launch_epikv_score(dtype, B, N, dm, hA, hB, window, (double)eps, g ? g : w.g, w.pre, scores, nullptr,
                            static_cast<cudaStream_t>(stream));
}

int kvc_epikv_evict(const kvc_cache* c, const void* hA, const void* hB, int32_t dm, int32_t window, float eps,
                    int32_t prefix, int32_t recent, const int32_t* budget, int32_t budget_all, int32_t* kept_idx,
                    int32_t* kept_len, float* scores, int32_t* status, void* workspace, size_t ws_bytes,
                    void* stream) {
  CacheGeom g;
  LayerPtrs K, V;
  int rc = check_cache(c, &g, &K, &V);
  if (rc) return rc;
  rc = check_epikv(c->dtype, c->B, c->N, dm, hA, hB, window, eps);
  if (rc) return rc;
  if (!kept_len || prefix < 0 || recent < 0) return KVC_ERR_INVALID_ARG;
  if (!budget && budget_all < prefix + recent && budget_all < c->N) return KVC_ERR_BUDGET_RANGE;
  if (!workspace || ws_bytes < epikv_ws(g.B, g.N, nullptr, nullptr) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return KVC_ERR_WORKSPACE;
  EpikvWs w;
  epikv_ws(g.B, g.N, &w, workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* sc = scores ? scores : w.scores;
  int32_t* ki = kept_idx ? kept_idx : w.kept;
  rc = launch_epikv_score(c->dtype, g.B, g.N, dm, hA, hB, window, (double)eps, w.g, w.pre, sc, w.keys, s);
  if (rc) return rc;
  // one selection per sequence on the order-preserving keys of the signed scores
  rc = launch_select(reinterpret_cast<const float*>(w.keys), g.B, g.N, prefix, recent, budget, budget_all, nullptr, 1,
                     ki, kept_len, status, s, true);
  if (rc) return rc;
  return launch_compact(g, c->dtype, K, V, ki, kept_len, status, false, s, true);
}

// ---------------------------------------------------------------------------
// kvc_score without a caller workspace: scratch lives in a fixed device region.
// ---------------------------------------------------------------------------
}  // extern "C"

namespace kvc {
namespace {
// The region every kvc_score_static call on a device uses (see kvc.h for sharing rules).
static __device__ __align__(256) unsigned char g_score_scratch[KVC_STATIC_SCRATCH_BYTES];

// Device address of the region in the current context (the symbol's name is only a host-side
// stand-in). Looked up on every call, not cached: a cached address would outlive the context it
// came from (after cudaDeviceReset, or a primary context released and made again) and point a
// launch at freed memory. The lookup is a table read once the module is loaded; the first one on
// a device loads the module, which is why the first call must come before any stream capture.
// NULL on failure.
void* static_scratch() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_score_scratch) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  return p;
}
}  // namespace
}  // namespace kvc

extern "C" int kvc_score_static(const kvc_cache* c, const void* q_recent, int32_t n_r, const void* qbuf,
                                const int32_t* count, int32_t qmax, int32_t n_b, int64_t t, double rope_theta,
                                float* scores, int32_t* beacon_picks, const kvc_opts* opts, void* stream) {
  CacheGeom g;
  LayerPtrs K, V;
  Opts o;
  int rc = check_cache(c, &g, &K, &V);
  if (rc) return rc;
  rc = check_opts(opts, false, &o);
  if (rc) return rc;
  rc = check_queries(c, q_recent, n_r, qbuf, count, qmax, n_b, rope_theta, o.ext);
  if (rc) return rc;
  if (!scores) return KVC_ERR_INVALID_ARG;
  const size_t need = score_ws_bytes(g, c->dtype, n_r, n_b, o.ext, nullptr, nullptr);
  if (need > (size_t)KVC_STATIC_SCRATCH_BYTES) return KVC_ERR_WORKSPACE;
  void* scratch = static_scratch();
  if (!scratch) return KVC_ERR_LAUNCH;
  ScoreWs ws;
  score_ws_bytes(g, c->dtype, n_r, n_b, o.ext, &ws, scratch);
  ScoreArgs a;
  fill_score_args(&a, g, c->dtype, K, q_recent, n_r, qbuf, count, qmax, n_b, t, rope_theta, scores, beacon_picks,
                  nullptr, o, o.entropy);
  return launch_score(a, ws, static_cast<cudaStream_t>(stream));
}
