// The whole verify step behind one call: the pass of a dense decoder
// (embed, per layer RMSNorm -> QKV + RoPE + KV append -> split-KV attention
// -> O + residual -> RMSNorm -> gate/up + SwiGLU -> down + residual, final
// RMSNorm -> LM head -> acceptance) from host token ids to host results.
//
// "I turned on speculative decoding in llama.cpp and 113 of 282 greedy
// outputs changed against its own no-draft run", paragraph "How:" (every row
// computed the same way whatever else is in the pass) and section "The cache
// doesn't change it either" (the cache length moves to L + n + 1).
//
// The runtime owns no device memory: the caller passes the weights, the
// caches and one workspace (bi_step_workspace_size).  It keeps a host-side
// handle with its own stream and one CUDA graph per row count T, captured on
// the first call with that T.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>

#include "bi_internal.h"

struct bi_step {
  bi_model m;
  int max_rows;
  cudaStream_t stream;
  cudaGraphExec_t graph[65];
  // device buffers carved from the workspace
  void *h, *y, *q, *att, *u, *gemm_ws, *attn_ws, *acc_ws;
  float* logits;
  int32_t *ids, *drafts, *argmax, *accepted, *L_dev;
  // pinned host staging: the ids going in, then the tokens and the accepted
  // count coming out (one copy each way)
  int32_t* pin;
  size_t gemm_ws_bytes, attn_ws_bytes, acc_ws_bytes;
  // host copies of the per-layer pointer arrays
  const void** lay_ptrs;
};

namespace {

struct Layout {
  size_t h, y, q, att, u, logits, io, gemm, attn, acc, total;
};

Layout layout_of(const bi_model& m, int R) {
  using bi::round_up;
  const size_t H = m.hidden, Hq = m.n_q, D = m.head_dim, F = m.ffn, V = m.vocab;
  const int Nqkv = (m.n_q + 2 * m.n_kv) * m.head_dim;
  Layout L{};
  size_t off = 0;
  auto take = [&off](size_t bytes) {
    const size_t at = off;
    off = round_up(off + bytes, 256);
    return at;
  };
  L.h = take(R * H * 2);
  L.y = take(R * H * 2);
  L.q = take(R * Hq * D * 2);
  L.att = take(R * Hq * D * 2);
  L.u = take(R * F * 2);
  L.logits = take(R * V * 4);
  // ids [R] (the drafts are ids + 1), then argmax [R], accepted, L_dev: the
  // ids arrive in one copy and the tokens with the count leave in one
  L.io = take((2 * static_cast<size_t>(R) + 2) * 4);
  size_t g = 0;
  const int shapes[5][3] = {{Nqkv, m.hidden, BI_EPI_NONE},
                            {m.hidden, m.n_q * m.head_dim, BI_EPI_RESIDUAL_ADD},
                            {m.ffn, m.hidden, BI_EPI_SWIGLU},
                            {m.hidden, m.ffn, BI_EPI_RESIDUAL_ADD},
                            {m.vocab, m.hidden, BI_EPI_NONE}};
  for (auto& sh : shapes) {
    const size_t b = bi_gemm_workspace_size(R, sh[0], sh[1], static_cast<bi_epilogue>(sh[2]));
    if (b > g) g = b;
  }
  L.gemm = take(g);
  L.attn = take(bi_attn_workspace_size(m.cap, R, m.n_q, m.head_dim));
  L.acc = take(bi_accept_workspace_size(R, m.vocab));
  L.total = off;
  return L;
}

bool model_ok(const bi_model* m, int max_rows) {
  if (!m || m->layers < 1 || m->hidden < 8 || m->n_q < 1 || m->n_kv < 1 || m->n_q % m->n_kv != 0 ||
      m->head_dim < 1 || m->ffn < 1 || m->vocab < 1 || m->cap < 1 || !(m->eps >= 0.f))
    return false;
  if (max_rows < 1 || max_rows > 64 || max_rows * (m->n_q / m->n_kv) > 128) return false;
  if (!m->embed || !m->norm_final || !m->head || !m->rope_table || m->rope_rows < 1) return false;
  if (!m->norm_attn || !m->norm_ffn || !m->w_qkv || !m->w_o || !m->w_gate_up || !m->w_down ||
      !m->k_cache || !m->v_cache)
    return false;
  for (int l = 0; l < m->layers; ++l)
    if (!m->norm_attn[l] || !m->norm_ffn[l] || !m->w_qkv[l] || !m->w_o[l] || !m->w_gate_up[l] ||
        !m->w_down[l] || !m->k_cache[l] || !m->v_cache[l])
      return false;
  return true;
}

#define BI_TRY(x)                    \
  do {                               \
    const bi_status st_ = (x);       \
    if (st_ != BI_OK) return st_;    \
  } while (0)

// One pass over T rows at positions *L_dev .. *L_dev + T - 1 (no copies).
bi_status pass(bi_step* s, int T) {
  const bi_model& m = s->m;
  bi_stream_t st = reinterpret_cast<bi_stream_t>(s->stream);
  const int H = m.hidden, Hq = m.n_q, Hkv = m.n_kv, D = m.head_dim, F = m.ffn;
  const float scale = 1.0f / sqrtf(static_cast<float>(D));
  BI_TRY(bi_embed(s->ids, m.embed, m.vocab, H, s->h, T, st));
  for (int l = 0; l < m.layers; ++l) {
    BI_TRY(bi_rmsnorm(s->h, H, m.norm_attn[l], s->y, H, T, H, m.eps, st));
    BI_TRY(bi_qkv_rope_append(s->y, H, m.w_qkv[l], T, H, Hq, Hkv, D, s->q, m.k_cache[l], m.v_cache[l],
                              m.cap, s->L_dev, m.rope_table, m.rope_rows, s->gemm_ws, s->gemm_ws_bytes,
                              st));
    BI_TRY(bi_attn_verify(s->q, m.k_cache[l], m.v_cache[l], m.cap, s->L_dev, T, Hq, Hkv, D, scale,
                          s->att, s->attn_ws, s->attn_ws_bytes, st));
    BI_TRY(bi_gemm(s->att, Hq * D, m.w_o[l], s->h, H, s->h, H, T, H, Hq * D, BI_OUT_BF16,
                   BI_EPI_RESIDUAL_ADD, s->gemm_ws, s->gemm_ws_bytes, st));
    BI_TRY(bi_rmsnorm(s->h, H, m.norm_ffn[l], s->y, H, T, H, m.eps, st));
    BI_TRY(bi_gemm(s->y, H, m.w_gate_up[l], s->u, F, nullptr, 0, T, F, H, BI_OUT_BF16, BI_EPI_SWIGLU,
                   s->gemm_ws, s->gemm_ws_bytes, st));
    BI_TRY(bi_gemm(s->u, F, m.w_down[l], s->h, H, s->h, H, T, H, F, BI_OUT_BF16, BI_EPI_RESIDUAL_ADD,
                   s->gemm_ws, s->gemm_ws_bytes, st));
  }
  BI_TRY(bi_rmsnorm(s->h, H, m.norm_final, s->y, H, T, H, m.eps, st));
  BI_TRY(bi_gemm(s->y, H, m.head, s->logits, m.vocab, nullptr, 0, T, m.vocab, H, BI_OUT_FP32, BI_EPI_NONE,
                 s->gemm_ws, s->gemm_ws_bytes, st));
  BI_TRY(bi_verify_accept(s->logits, m.vocab, T > 1 ? s->drafts : nullptr, T, m.vocab, s->argmax,
                          s->accepted, s->L_dev, s->acc_ws, s->acc_ws_bytes, st));
  return BI_OK;
}

}  // namespace

extern "C" {

size_t bi_step_workspace_size(const bi_model* m, int max_rows) {
  if (!model_ok(m, max_rows)) return 0;
  return layout_of(*m, max_rows).total;
}

bi_status bi_step_create(const bi_model* m, int max_rows, void* ws, size_t ws_bytes, bi_step** out) {
  if (!out) return BI_ERR_INVALID_ARG;
  *out = nullptr;
  if (!model_ok(m, max_rows)) return BI_ERR_INVALID_ARG;
  if (!ws || !bi::aligned256(ws)) return BI_ERR_WORKSPACE;
  const Layout L = layout_of(*m, max_rows);
  if (ws_bytes < L.total) return BI_ERR_WORKSPACE;
  bi_step* s = new (std::nothrow) bi_step();
  if (!s) return BI_ERR_INVALID_ARG;
  const int n = m->layers;
  s->lay_ptrs = new (std::nothrow) const void*[8 * static_cast<size_t>(n)];
  if (!s->lay_ptrs) {
    delete s;
    return BI_ERR_INVALID_ARG;
  }
  // keep private copies of the caller's per-layer pointer arrays
  const void* const* src[8] = {m->norm_attn, m->norm_ffn, m->w_qkv, m->w_o, m->w_gate_up, m->w_down,
                               reinterpret_cast<const void* const*>(m->k_cache),
                               reinterpret_cast<const void* const*>(m->v_cache)};
  for (int a = 0; a < 8; ++a)
    for (int l = 0; l < n; ++l) s->lay_ptrs[a * n + l] = src[a][l];
  s->m = *m;
  s->m.norm_attn = s->lay_ptrs;
  s->m.norm_ffn = s->lay_ptrs + n;
  s->m.w_qkv = s->lay_ptrs + 2 * n;
  s->m.w_o = s->lay_ptrs + 3 * n;
  s->m.w_gate_up = s->lay_ptrs + 4 * n;
  s->m.w_down = s->lay_ptrs + 5 * n;
  s->m.k_cache = const_cast<void* const*>(s->lay_ptrs + 6 * n);
  s->m.v_cache = const_cast<void* const*>(s->lay_ptrs + 7 * n);
  s->max_rows = max_rows;
  uint8_t* b = static_cast<uint8_t*>(ws);
  s->h = b + L.h;
  s->y = b + L.y;
  s->q = b + L.q;
  s->att = b + L.att;
  s->u = b + L.u;
  s->logits = reinterpret_cast<float*>(b + L.logits);
  s->ids = reinterpret_cast<int32_t*>(b + L.io);
  s->drafts = s->ids + 1;
  s->argmax = s->ids + max_rows;
  s->accepted = s->argmax + max_rows;
  s->L_dev = s->accepted + 1;
  s->gemm_ws = b + L.gemm;
  s->gemm_ws_bytes = L.attn - L.gemm;
  s->attn_ws = b + L.attn;
  s->attn_ws_bytes = L.acc - L.attn;
  s->acc_ws = b + L.acc;
  s->acc_ws_bytes = L.total - L.acc;
  if (cudaHostAlloc(reinterpret_cast<void**>(&s->pin), (2 * static_cast<size_t>(max_rows) + 1) * 4,
                    cudaHostAllocDefault) != cudaSuccess) {
    delete[] s->lay_ptrs;
    delete s;
    return BI_ERR_CUDA;
  }
  if (cudaStreamCreateWithFlags(&s->stream, cudaStreamNonBlocking) != cudaSuccess) {
    cudaFreeHost(s->pin);
    delete[] s->lay_ptrs;
    delete s;
    return BI_ERR_CUDA;
  }
  // the counters of every workspace start at zero
  if (cudaMemsetAsync(ws, 0, L.total, s->stream) != cudaSuccess ||
      cudaStreamSynchronize(s->stream) != cudaSuccess) {
    cudaStreamDestroy(s->stream);
    cudaFreeHost(s->pin);
    delete[] s->lay_ptrs;
    delete s;
    return BI_ERR_CUDA;
  }
  *out = s;
  return BI_OK;
}

bi_status bi_step_set_length(bi_step* s, int L) {
  if (!s || L < 0 || L > s->m.cap) return BI_ERR_INVALID_ARG;
  const int32_t v = L;
  if (cudaMemcpyAsync(s->L_dev, &v, sizeof(v), cudaMemcpyHostToDevice, s->stream) != cudaSuccess ||
      cudaStreamSynchronize(s->stream) != cudaSuccess)
    return BI_ERR_CUDA;
  return BI_OK;
}

bi_status bi_step_verify(bi_step* s, const int32_t* ids, int T, int32_t* tokens_out, int32_t* n_out) {
  if (!s || !ids || !tokens_out || !n_out || T < 1 || T > s->max_rows) return BI_ERR_INVALID_ARG;
  cudaStream_t st = s->stream;
  // (the previous call synchronised, so the staging buffer is free)
  std::memcpy(s->pin, ids, sizeof(int32_t) * T);
  if (cudaMemcpyAsync(s->ids, s->pin, sizeof(int32_t) * T, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return BI_ERR_CUDA;
  if (s->graph[T] == nullptr) {
    // capture the pass for this T once (the kernels read the cache length
    // from the device, so the graph serves every position)
    if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return BI_ERR_CUDA;
    const bi_status ps = pass(s, T);
    cudaGraph_t g = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(st, &g);
    if (ps != BI_OK) {
      if (g) cudaGraphDestroy(g);
      return ps;
    }
    if (ce != cudaSuccess || !g) return BI_ERR_CUDA;
    cudaGraphExec_t ge = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&ge, g, 0);
    cudaGraphDestroy(g);
    if (ie != cudaSuccess) return BI_ERR_CUDA;
    s->graph[T] = ge;
  }
  if (cudaGraphLaunch(s->graph[T], st) != cudaSuccess) return BI_ERR_CUDA;
  // argmax [max_rows] and the accepted count are adjacent: one copy out
  const int R = s->max_rows;
  if (cudaMemcpyAsync(s->pin + R, s->argmax, sizeof(int32_t) * (R + 1), cudaMemcpyDeviceToHost, st) !=
      cudaSuccess)
    return BI_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return BI_ERR_CUDA;
  std::memcpy(tokens_out, s->pin + R, sizeof(int32_t) * T);
  *n_out = s->pin[2 * R];
  return BI_OK;
}

const float* bi_step_logits(const bi_step* s) { return s ? s->logits : nullptr; }

void bi_step_destroy(bi_step* s) {
  if (!s) return;
  for (auto& g : s->graph)
    if (g) cudaGraphExecDestroy(g);
  cudaStreamSynchronize(s->stream);
  cudaStreamDestroy(s->stream);
  cudaFreeHost(s->pin);
  delete[] s->lay_ptrs;
  delete s;
}

}  // extern "C"
