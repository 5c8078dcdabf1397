// spec_abi.cu -- the extern "C" entry points of libspec_verify.so: argument checks on the host,
// workspace layout, launch configuration, and dispatch to the kernel instances.
#include <cuda_runtime.h>
#include <float.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include "spec_launch.h"
#include "spec_verify.h"

using namespace specv;

namespace {

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices];   // cached multiprocessor counts (0 = not queried yet)

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
  if (dev < kMaxDevices && g_sm_count[dev] > 0) return g_sm_count[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev < kMaxDevices) g_sm_count[dev] = n;
  return n;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

int elem_size(int dtype) { return dtype == SPEC_BF16 ? 2 : 4; }

// units per logits row: one unit is 32 lanes x 8 vectors of 16 bytes
int chunks_per_row(int V, int dtype) {
  const int epv = 16 / elem_size(dtype);
  const long long nv = V / epv;
  const long long c = (nv + kUnitVecs - 1) / kUnitVecs;
  return c < 1 ? 1 : static_cast<int>(c);
}

struct Layout {
  size_t part, xlogit, total;
};

// workspace: [unit partials | draft-token logits], each part 256-byte aligned
Layout layout(long long B, long long R, long long C) {
  Layout L;
  L.part = 0;
  L.xlogit = L.part + align256(static_cast<size_t>(B * R * C) * 8);
  L.total = L.xlogit + align256(static_cast<size_t>(B * R) * 4);
  return L;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool temp_ok(float T) { return T == 0.f || (T >= FLT_MIN && T <= FLT_MAX); }

// Fills the unit counts of p; returns SPEC_OK, or SPEC_ERR_SHAPE when the call has 2^31 - 64
// units or more (unit ids are 32-bit on the device).
int plan_units(Params &p, int dtype) {
  p.C = chunks_per_row(p.V, dtype);
  const long long units = static_cast<long long>(p.B) * p.R * p.C;
  if (units >= (1LL << 31) - 64) return SPEC_ERR_SHAPE;
  p.units = static_cast<int>(units);
  p.upb = p.R * p.C;
  return SPEC_OK;
}

// plan_units, then the workspace pointers; SPEC_ERR_WORKSPACE when the workspace is too small.
int plan(Params &p, int dtype, void *ws, size_t ws_bytes) {
  const int rc = plan_units(p, dtype);
  if (rc != SPEC_OK) return rc;
  const Layout L = layout(p.B, p.R, p.C);
  if (ws_bytes < L.total) return SPEC_ERR_WORKSPACE;
  char *w = static_cast<char *>(ws);
  p.ws_part = reinterpret_cast<uint2 *>(w + L.part);
  p.ws_xlogit = reinterpret_cast<float *>(w + L.xlogit);
  return SPEC_OK;
}

// Stream kernel grid: two CTAs of 512 threads per SM (all resident at once), never more CTAs
// than groups of kWarps units. (Trimming the grid so that the last round of loads is full, and
// one CTA per SM streaming through a cp.async ring in shared memory, were both measured slower.)
int grid_for(const Params &p) {
  const long long cap = 2LL * (sm_count() > 0 ? sm_count() : 1);
  const long long groups = (static_cast<long long>(p.units) + kWarps - 1) / kWarps;
  long long g = groups < cap ? groups : cap;
  return g < 1 ? 1 : static_cast<int>(g);
}

// Finishing plan for chain sampling. Single-unit rows with gamma <= 31: one warp per batch row.
// Otherwise one cluster of S CTAs per batch row: S is the largest power of two (at most 8) for
// which all B*S CTAs are resident at once (two per SM) and every CTA gets at least 8 residual
// segments.
FinishPlan chain_sample_plan(const Params &p, int dtype) {
  FinishPlan f{};
  if (p.C == 1 && p.V <= kWarpTailMaxV && p.gamma <= 31) {
    f.warp_tail = true;
    f.cluster = 1;
    f.grid = (p.B + kTailWarpsPerCta - 1) / kTailWarpsPerCta;
    f.smem = 0;
    return f;
  }
  // Sampling (no drafts) with every row on a 16-byte boundary: the draw needs only the row's
  // unit partials and one unit, which one warp does (its C partials staged in shared memory).
  const bool rows_aligned = (reinterpret_cast<uintptr_t>(p.tgt) & 15u) == 0 &&
                            (static_cast<long long>(p.V) * elem_size(dtype)) % 16 == 0;
  if (p.gamma == 0 && rows_aligned) {
    f.sample_warp = true;
    f.cluster = 1;
    f.grid = (p.B + kTailWarpsPerCta - 1) / kTailWarpsPerCta;
    f.smem = sizeof(uint2) * static_cast<size_t>(kTailWarpsPerCta) * static_cast<size_t>(p.C);
    return f;
  }
  const int nseg = (p.V + kSeg - 1) / kSeg;
  const int sms = sm_count() > 0 ? sm_count() : 1;
  int cap = nseg / 8;
  if (cap > kMaxCluster) cap = kMaxCluster;
  const int fit = (2 * sms) / p.B;
  if (cap > fit) cap = fit;
  int S = 1;
  while (2 * S <= cap) S *= 2;
  f.warp_tail = false;
  f.cluster = S;
  f.grid = p.B * S;
  // rowM, rowZ (2R floats: 8-byte aligned end), the bonus row's unit partials, the segment sums
  f.smem = sizeof(float) * 2 * static_cast<size_t>(p.R) +
           sizeof(uint2) * static_cast<size_t>(p.C) + sizeof(float) * nseg;
  return f;
}

FinishPlan cta_plan(int rows, size_t smem) {
  FinishPlan f{};
  f.grid = rows;
  f.cluster = 1;
  f.smem = smem;
  f.warp_tail = false;
  return f;
}

Params blank() {
  Params p{};
  return p;
}

float c2_of(float T) {
  return T == 0.f ? 0.f : static_cast<float>(1.4426950408889634 / static_cast<double>(T));
}

// Row geometry of each kind of call (no pointers).
void chain_shape(Params &p, int B, int gamma, int V, float T) {
  const bool greedy = T == 0.f;
  p.B = B;
  p.gamma = gamma;
  p.N = 0;
  p.V = V;
  p.Rt = gamma + 1;
  p.Rd = greedy ? 0 : gamma;
  p.R = p.Rt + p.Rd;
  p.c2 = c2_of(T);
}

void tree_shape(Params &p, int B, int N, int V) {
  p.B = B;
  p.N = N;
  p.V = V;
  p.Rt = N;
  p.Rd = 0;
  p.R = N;
}

void probs_shape(Params &p, int rows, int V, float T) {
  p.B = rows;
  p.V = V;
  p.Rt = 1;
  p.Rd = 0;
  p.R = 1;
  p.c2 = c2_of(T);
}

// The launch plan of each kind of call (after plan_units).
FinishPlan chain_finish(const Params &p, bool greedy, int dtype) {
  return greedy ? cta_plan(p.B, sizeof(int) * (2 * static_cast<size_t>(p.R) + p.gamma))
                : chain_sample_plan(p, dtype);
}

FinishPlan tree_finish(const Params &p) {
  return cta_plan(p.B, sizeof(int) * 6 * static_cast<size_t>(p.N));
}

// Probabilities: row-resident (one kernel; a cluster of S CTAs per row, S the fewest that hold
// the row's interior in registers) when S <= kMaxCluster, else the stream kernel plus the
// unit-granular write pass.
FinishPlan probs_finish(const Params &p, int dtype) {
  const int epv = 16 / elem_size(dtype);
  const long long quads = static_cast<long long>(p.V / epv) * epv / 4;
  const long long cap = static_cast<long long>(kThreads) *
                        (dtype == SPEC_BF16 ? kResQuads<uint16_t> : kResQuads<float>);
  const long long S = quads > 0 ? (quads + cap - 1) / cap : 1;
  if (S <= kMaxCluster) {
    FinishPlan f{};
    f.resident = true;
    f.cluster = static_cast<int>(S);
    f.grid = p.B * f.cluster;
    return f;
  }
  return cta_plan(grid_for(p), 0);
}

}  // namespace

namespace specv {

// The CUDA error behind the last SPEC_ERR_LAUNCH returned on this thread (spec_last_cuda_error).
thread_local int g_last_cuda_error = 0;

int launch_result(cudaError_t e) {
  if (e == cudaSuccess) return SPEC_OK;
  g_last_cuda_error = static_cast<int>(e);
  return SPEC_ERR_LAUNCH;
}

// The host checks of a chain call, in the order the header documents: dtype, shape,
// temperature, null pointers, alignment. The workspace is checked only when asked (the
// static-scratch entry point has none); nothing here needs a device.
int chain_args_check(const void *target_logits, const void *draft_logits, int dtype,
                     const int32_t *draft_tokens, const float *uniforms, int B, int gamma, int V,
                     float temperature, const int32_t *accept_len, const int32_t *out_tokens,
                     const int32_t *status, const void *workspace, bool need_workspace) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (B < 0 || gamma < 0 || gamma > SPEC_MAX_GAMMA || V < 1 || V > SPEC_MAX_V)
    return SPEC_ERR_SHAPE;
  if (!temp_ok(temperature)) return SPEC_ERR_TEMP;
  const bool greedy = temperature == 0.f;
  if (!target_logits || !accept_len || !out_tokens || !status || (need_workspace && !workspace))
    return SPEC_ERR_NULL;
  if (gamma > 0 && !draft_tokens) return SPEC_ERR_NULL;
  if (!greedy && (!uniforms || (gamma > 0 && !draft_logits))) return SPEC_ERR_NULL;
  const int es = elem_size(dtype);
  if (!aligned(target_logits, es) || (draft_logits && !aligned(draft_logits, es)) ||
      (draft_tokens && !aligned(draft_tokens, 4)) || (uniforms && !aligned(uniforms, 4)) ||
      !aligned(accept_len, 4) || !aligned(out_tokens, 4) || !aligned(status, 4) ||
      (need_workspace && !aligned(workspace, 16)))
    return SPEC_ERR_ALIGN;
  return SPEC_OK;
}

// The bounded-wait self-check kernel's launcher (spec_lmhead.cu, beside the kernel whose waits it
// exercises): one cluster of two CTAs.
cudaError_t launch_wait_selftest(int32_t *status, unsigned long long limit_ns,
                                 cudaStream_t stream);
}  // namespace specv

extern "C" {

size_t spec_workspace_bytes(int B, int rows_per_b, int V, int dtype) {
  if (B < 0 || rows_per_b < 1 || V < 1 || V > SPEC_MAX_V) return 0;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return 0;
  return layout(B, rows_per_b, chunks_per_row(V, dtype)).total;
}

int spec_workspace_init(void *workspace, size_t workspace_bytes, void *stream) {
  if (!workspace) return SPEC_ERR_NULL;
  if (!aligned(workspace, 16)) return SPEC_ERR_ALIGN;
  return specv::launch_result(
      cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)));
}

int spec_verify_chain(const void *target_logits, const void *draft_logits, int dtype,
                      const int32_t *draft_tokens, const float *uniforms, int B, int gamma, int V,
                      float temperature, int32_t *accept_len, int32_t *out_tokens,
                      int32_t *status, void *workspace, size_t workspace_bytes, void *stream) {
  const int chk = specv::chain_args_check(target_logits, draft_logits, dtype, draft_tokens,
                                          uniforms, B, gamma, V, temperature, accept_len,
                                          out_tokens, status, workspace, true);
  if (chk != SPEC_OK) return chk;
  const bool greedy = temperature == 0.f;
  if (B == 0) return SPEC_OK;

  Params p = blank();
  chain_shape(p, B, gamma, V, temperature);
  p.tgt = target_logits;
  p.drf = greedy ? nullptr : draft_logits;
  p.tokens = draft_tokens;
  p.uniforms = greedy ? nullptr : uniforms;
  p.accept_len = accept_len;
  p.out_tokens = out_tokens;
  p.status = status;
  const int rc = plan(p, dtype, workspace, workspace_bytes);
  if (rc != SPEC_OK) return rc;
  const FinishPlan f = chain_finish(p, greedy, dtype);
  const cudaError_t e = launch_chain(greedy ? kChainGreedy : kChainSample, dtype, p, grid_for(p),
                                     f, static_cast<cudaStream_t>(stream));
  return specv::launch_result(e);
}

int spec_verify_tree(const void *target_logits, int dtype, const int32_t *parents,
                     const int32_t *node_tokens, int B, int N, int V, int32_t *accept_len,
                     int32_t *path_nodes, int32_t *out_tokens, int32_t *status,
                     void *workspace, size_t workspace_bytes, void *stream) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (B < 0 || N < 1 || N > SPEC_MAX_NODES || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_SHAPE;
  if (!target_logits || !parents || !node_tokens || !accept_len || !path_nodes || !out_tokens ||
      !status || !workspace)
    return SPEC_ERR_NULL;
  if (!aligned(target_logits, elem_size(dtype)) || !aligned(parents, 4) ||
      !aligned(node_tokens, 4) || !aligned(accept_len, 4) || !aligned(path_nodes, 4) ||
      !aligned(out_tokens, 4) || !aligned(status, 4) || !aligned(workspace, 16))
    return SPEC_ERR_ALIGN;
  if (B == 0) return SPEC_OK;

  Params p = blank();
  tree_shape(p, B, N, V);
  p.tgt = target_logits;
  p.tokens = node_tokens;
  p.parents = parents;
  p.accept_len = accept_len;
  p.out_tokens = out_tokens;
  p.path_nodes = path_nodes;
  p.status = status;
  const int rc = plan(p, dtype, workspace, workspace_bytes);
  if (rc != SPEC_OK) return rc;
  const FinishPlan f = tree_finish(p);
  const cudaError_t e = launch_tree(dtype, p, grid_for(p), f, static_cast<cudaStream_t>(stream));
  return specv::launch_result(e);
}

size_t spec_lmhead_workspace_bytes(int B, int gamma, int V) {
  if (B < 0 || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 256 || V % 256 ||
      V > SPEC_LMHEAD_MAX_V)
    return 0;
  return layout(B, 2LL * gamma + 1, V / 256).total;
}

int spec_verify_chain_lmhead(const void *hidden_t, const void *head_t, int hidden_t_size,
                             const void *hidden_d, const void *head_d, int hidden_d_size,
                             const int32_t *draft_tokens,
                             const float *uniforms, int B, int gamma, int V, float temperature,
                             void *logits_t, void *logits_d, int32_t *accept_len,
                             int32_t *out_tokens, int32_t *status, void *workspace,
                             size_t workspace_bytes, void *stream) {
  if (B < 0 || gamma < 1 || gamma > SPEC_MAX_GAMMA || V < 256 || V % 256 ||
      V > SPEC_LMHEAD_MAX_V || hidden_t_size < 64 || hidden_t_size % 64 || hidden_d_size < 64 ||
      hidden_d_size % 64 ||
      static_cast<long long>(B) * (2 * gamma + 1) * (V / 256) > INT_MAX)
    return SPEC_ERR_SHAPE;
  if (!(temperature >= FLT_MIN && temperature <= FLT_MAX)) return SPEC_ERR_TEMP;
  if (!hidden_t || !head_t || !hidden_d || !head_d || !draft_tokens || !uniforms || !logits_t ||
      !logits_d || !accept_len || !out_tokens || !status || !workspace)
    return SPEC_ERR_NULL;
  if (!aligned(hidden_t, 16) || !aligned(head_t, 16) || !aligned(hidden_d, 16) ||
      !aligned(head_d, 16) || !aligned(logits_t, 16) || !aligned(logits_d, 16) ||
      !aligned(draft_tokens, 4) || !aligned(uniforms, 4) || !aligned(accept_len, 4) ||
      !aligned(out_tokens, 4) || !aligned(status, 4) || !aligned(workspace, 16))
    return SPEC_ERR_ALIGN;
  if (B == 0) return SPEC_OK;
  Params p = blank();
  chain_shape(p, B, gamma, V, temperature);
  p.tgt = logits_t;   // written by the producer, re-read by the draw
  p.drf = logits_d;
  p.tokens = draft_tokens;
  p.uniforms = uniforms;
  p.accept_len = accept_len;
  p.out_tokens = out_tokens;
  p.status = status;
  p.tile_units = 1;
  p.C = V / 256;   // one partial per 256-column tile of a row
  p.upb = p.R * p.C;
  p.units = static_cast<int>(static_cast<long long>(B) * p.upb);
  const Layout L = layout(B, p.R, p.C);
  if (workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  p.ws_part = reinterpret_cast<uint2 *>(static_cast<char *>(workspace) + L.part);
  p.ws_xlogit = reinterpret_cast<float *>(static_cast<char *>(workspace) + L.xlogit);
  const FinishPlan f = chain_sample_plan(p, SPEC_BF16);
  const cudaError_t e =
      launch_lmhead(p, hidden_t, head_t, hidden_t_size, hidden_d, head_d, hidden_d_size, logits_t,
                    logits_d, f, static_cast<cudaStream_t>(stream));
  return specv::launch_result(e);
}

int spec_verify_tree_sample(const void *target_logits, const void *draft_logits, int dtype,
                            const int32_t *parents, const int32_t *node_tokens,
                            const float *uniforms, int B, int N, int V, float temperature,
                            int32_t *accept_len, int32_t *path_nodes, int32_t *out_tokens,
                            int32_t *status, void *workspace, size_t workspace_bytes,
                            void *stream) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (B < 0 || N < 1 || N > SPEC_MAX_NODES || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_SHAPE;
  if (!temp_ok(temperature)) return SPEC_ERR_TEMP;
  if (temperature == 0.f)   // greedy: the argmax walk, draft logits and uniforms not read
    return spec_verify_tree(target_logits, dtype, parents, node_tokens, B, N, V, accept_len,
                            path_nodes, out_tokens, status, workspace, workspace_bytes, stream);
  if (!target_logits || !draft_logits || !parents || !node_tokens || !uniforms || !accept_len ||
      !path_nodes || !out_tokens || !status || !workspace)
    return SPEC_ERR_NULL;
  const int es = elem_size(dtype);
  if (!aligned(target_logits, es) || !aligned(draft_logits, es) || !aligned(parents, 4) ||
      !aligned(node_tokens, 4) || !aligned(uniforms, 4) || !aligned(accept_len, 4) ||
      !aligned(path_nodes, 4) || !aligned(out_tokens, 4) || !aligned(status, 4) ||
      !aligned(workspace, 16))
    return SPEC_ERR_ALIGN;
  if (B == 0) return SPEC_OK;
  Params p = blank();
  p.B = B;
  p.N = N;
  p.V = V;
  p.Rt = N;   // rows 0 .. N-1: target; N .. 2N-1: draft
  p.Rd = N;
  p.R = 2 * N;
  p.c2 = c2_of(temperature);
  p.tgt = target_logits;
  p.drf = draft_logits;
  p.parents = parents;
  p.tokens = node_tokens;
  p.uniforms = uniforms;
  p.accept_len = accept_len;
  p.path_nodes = path_nodes;
  p.out_tokens = out_tokens;
  p.status = status;
  const int rc = plan(p, dtype, workspace, workspace_bytes);
  if (rc != SPEC_OK) return rc;
  // rowM, rowZ [2N] floats; parents, tokens, children [N] ints; segment sums
  const size_t smem = sizeof(float) * 4 * static_cast<size_t>(N) +
                      sizeof(int) * 3 * static_cast<size_t>(N) +
                      sizeof(float) * static_cast<size_t>((V + kSeg - 1) / kSeg);
  const cudaError_t e = launch_tree_sample(dtype, p, grid_for(p), smem,
                                           static_cast<cudaStream_t>(stream));
  return specv::launch_result(e);
}

int spec_probs(const void *logits, int dtype, int rows, int V, float temperature,
               float *out_probs, int32_t *status, void *workspace, size_t workspace_bytes,
               void *stream) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (rows < 0 || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_SHAPE;
  if (!temp_ok(temperature)) return SPEC_ERR_TEMP;
  if (!logits || !out_probs || !status || !workspace) return SPEC_ERR_NULL;
  if (!aligned(logits, elem_size(dtype)) || !aligned(out_probs, 4) || !aligned(status, 4) ||
      !aligned(workspace, 16))
    return SPEC_ERR_ALIGN;
  if (rows == 0) return SPEC_OK;
  const bool greedy = temperature == 0.f;
  Params p = blank();
  probs_shape(p, rows, V, temperature);
  p.tgt = logits;
  p.out_probs = out_probs;
  p.status = status;
  const int rc = plan(p, dtype, workspace, workspace_bytes);
  if (rc != SPEC_OK) return rc;
  const cudaError_t e = launch_probs(greedy ? kProbsGreedy : kProbs, dtype, p, grid_for(p),
                                     probs_finish(p, dtype), static_cast<cudaStream_t>(stream));
  return specv::launch_result(e);
}

int spec_sample(const void *logits, int dtype, int rows, int V, float temperature,
                const float *uniforms, int32_t *out_tokens, int32_t *status, void *workspace,
                size_t workspace_bytes, void *stream) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (rows < 0 || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_SHAPE;
  if (!temp_ok(temperature)) return SPEC_ERR_TEMP;
  const bool greedy = temperature == 0.f;
  if (!logits || !out_tokens || !status || !workspace || (!greedy && !uniforms))
    return SPEC_ERR_NULL;
  if (!aligned(logits, elem_size(dtype)) || (uniforms && !aligned(uniforms, 4)) ||
      !aligned(out_tokens, 4) || !aligned(status, 4) || !aligned(workspace, 16))
    return SPEC_ERR_ALIGN;
  if (rows == 0) return SPEC_OK;
  // a chain step with no drafts: the bonus draw from each row (argmax at T == 0)
  Params p = blank();
  chain_shape(p, rows, 0, V, temperature);
  p.tgt = logits;
  p.uniforms = greedy ? nullptr : uniforms;
  p.accept_len = nullptr;
  p.out_tokens = out_tokens;
  p.status = status;
  const int rc = plan(p, dtype, workspace, workspace_bytes);
  if (rc != SPEC_OK) return rc;
  const FinishPlan f = chain_finish(p, greedy, dtype);
  const cudaError_t e = launch_chain(greedy ? kChainGreedy : kChainSample, dtype, p, grid_for(p),
                                     f, static_cast<cudaStream_t>(stream));
  return specv::launch_result(e);
}

int spec_topk(const void *logits, int dtype, int rows, int V, int k, int32_t *out_idx,
              int32_t *status, void *workspace, size_t workspace_bytes, void *stream) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (rows < 0 || V < 1 || V > SPEC_MAX_V || k < 1 || k > SPEC_MAX_TOPK || k > V)
    return SPEC_ERR_SHAPE;
  if (!logits || !out_idx || !status || !workspace) return SPEC_ERR_NULL;
  if (!aligned(logits, elem_size(dtype)) || !aligned(out_idx, 4) || !aligned(status, 4) ||
      !aligned(workspace, 16))
    return SPEC_ERR_ALIGN;
  if (rows == 0) return SPEC_OK;
  Params p = blank();
  probs_shape(p, rows, V, 1.f);
  p.tgt = logits;
  p.out_tokens = out_idx;
  p.status = status;
  p.topk = k;
  const int rc = plan_units(p, dtype);
  if (rc != SPEC_OK) return rc;
  // k candidates (8 bytes each) per unit: the unit partials region of a call with k rows per row
  if (workspace_bytes < layout(rows, k, p.C).total) return SPEC_ERR_WORKSPACE;
  p.ws_part = static_cast<uint2 *>(workspace);
  // one CTA of 512 threads per SM (up to 128 registers per thread for the lists)
  const long long cap = sm_count() > 0 ? sm_count() : 1;
  const long long groups = (static_cast<long long>(p.units) + kWarps - 1) / kWarps;
  const int grid = static_cast<int>(groups < cap ? groups : cap);
  const cudaError_t e = launch_topk(dtype, p, grid < 1 ? 1 : grid,
                                    static_cast<cudaStream_t>(stream));
  return specv::launch_result(e);
}

int spec_tree_mask(const int32_t *parents, int B, int N, uint32_t *mask_words, int32_t *status,
                   void *stream) {
  if (B < 0 || N < 1 || N > SPEC_MAX_NODES) return SPEC_ERR_SHAPE;
  if (!parents || !mask_words || !status) return SPEC_ERR_NULL;
  if (!aligned(parents, 4) || !aligned(mask_words, 4) || !aligned(status, 4))
    return SPEC_ERR_ALIGN;
  if (B == 0) return SPEC_OK;
  Params p = blank();
  p.parents = parents;
  p.mask_words = mask_words;
  p.status = status;
  p.B = B;
  p.N = N;
  const cudaError_t e = launch_tree_mask(p, static_cast<cudaStream_t>(stream));
  return specv::launch_result(e);
}

int spec_launch_shape(int kind, int B, int rows_per_b, int V, int dtype, float temperature,
                      int *kernels, int *grid, int *cluster) {
  if (!kernels || !grid || !cluster) return SPEC_ERR_NULL;
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_DTYPE;
  if (B < 1 || rows_per_b < 1 || V < 1 || V > SPEC_MAX_V) return SPEC_ERR_SHAPE;
  Params p = blank();
  FinishPlan f{};
  if (kind == SPEC_CALL_CHAIN) {
    if (!temp_ok(temperature)) return SPEC_ERR_TEMP;
    if ((rows_per_b & 1) == 0 || (rows_per_b - 1) / 2 > SPEC_MAX_GAMMA) return SPEC_ERR_SHAPE;
    chain_shape(p, B, (rows_per_b - 1) / 2, V, temperature);
    const int rc = plan_units(p, dtype);
    if (rc != SPEC_OK) return rc;
    f = chain_finish(p, temperature == 0.f, dtype);
  } else if (kind == SPEC_CALL_TREE) {
    if (rows_per_b > SPEC_MAX_NODES) return SPEC_ERR_SHAPE;
    tree_shape(p, B, rows_per_b, V);
    const int rc = plan_units(p, dtype);
    if (rc != SPEC_OK) return rc;
    f = tree_finish(p);
  } else if (kind == SPEC_CALL_PROBS) {
    if (!temp_ok(temperature)) return SPEC_ERR_TEMP;
    if (rows_per_b != 1) return SPEC_ERR_SHAPE;
    probs_shape(p, B, V, temperature);
    const int rc = plan_units(p, dtype);
    if (rc != SPEC_OK) return rc;
    f = probs_finish(p, dtype);
  } else {
    return SPEC_ERR_SHAPE;
  }
  *kernels = f.resident ? 1 : 2;
  *grid = f.grid;
  *cluster = f.cluster;
  return SPEC_OK;
}

int spec_selftest_bounded_wait(int32_t *status, double limit_seconds, void *stream) {
  if (!status) return SPEC_ERR_NULL;
  if (!aligned(status, 4)) return SPEC_ERR_ALIGN;
  if (!(limit_seconds >= 1e-6 && limit_seconds <= 10.0)) return SPEC_ERR_SHAPE;
  const auto ns = static_cast<unsigned long long>(limit_seconds * 1e9);
  return specv::launch_result(
      specv::launch_wait_selftest(status, ns, static_cast<cudaStream_t>(stream)));
}

int spec_last_cuda_error(void) { return specv::g_last_cuda_error; }

const char *spec_cuda_error_string(int cuda_error) {
  return cudaGetErrorString(static_cast<cudaError_t>(cuda_error));
}

const char *spec_status_string(int code) {
  switch (code) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_NULL: return "a required pointer is NULL";
    case SPEC_ERR_SHAPE: return "B, gamma, N, V or rows out of range";
    case SPEC_ERR_TEMP: return "temperature must be 0 or a finite value >= FLT_MIN";
    case SPEC_ERR_DTYPE: return "dtype must be SPEC_F32 or SPEC_BF16";
    case SPEC_ERR_WORKSPACE: return "workspace smaller than spec_workspace_bytes()";
    case SPEC_ERR_ALIGN: return "pointer not aligned to its element size (workspace: 16 bytes)";
    case SPEC_ERR_LAUNCH: return "kernel launch failed";
    case SPEC_ERR_NONFINITE: return "a logits row holds NaN or +inf, or no finite value";
    case SPEC_ERR_TOKEN: return "a draft or node token is outside [0, V)";
    case SPEC_ERR_PARENT: return "a tree parent index is invalid";
    case SPEC_ERR_CHECK: return "checked build: a computed index fell outside its buffer";
    case SPEC_ERR_TIMEOUT: return "a bounded wait inside a kernel gave up";
    default: return "unknown status";
  }
}

}  // extern "C"
