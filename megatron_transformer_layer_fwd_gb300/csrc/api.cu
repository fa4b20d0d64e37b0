// C ABI (include/mgb.h): argument validation, buffer plans, and the launch
// sequences of the layer forward/backward and the chunked cross-entropy.
//
// Layer dataflow: "LLM Lab 06: build a Megatron-style Transformer Block from
// scratch", section 2 (LN -> attention -> residual -> LN -> fc1 -> GELU -> fc2
// -> residual, loss = mean(out), end-to-end backward) and section 5 (Post-LN
// moves the norm after each residual add); "02 - How a whole Transformer block
// is split", sections 1-2 (SwiGLU interleave, fused QKV, GQA, output
// projection) and sections 3-4 (tied embedding, chunked cross-entropy).
// On one GPU the tensor-parallel all-gather / all-reduce points of those pages
// disappear: each head writes its own column slice of the attention output and
// the row-parallel partial sums are the K loop of the projection / fc2 GEMMs.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <memory>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mgb {

// One error word per device that loads the library (see mgb_device_status).
__device__ int g_error_word = 0;

void* current_cuda_context() {
  typedef int (*GetCurrent)(void**);  // cuCtxGetCurrent(CUcontext*)
  static GetCurrent fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<GetCurrent>(f);
  });
  void* ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != 0) return nullptr;
  return ctx;
}

int* device_error_word() {
  // looked up once per device and context (a reset device gets a new one)
  static int* addr[64] = {};
  static void* ctx_of[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  void* ctx = current_cuda_context();
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || ctx == nullptr || ctx_of[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(p);
    ctx_of[dev] = current_cuda_context();  // the lookup made the context current
  }
  return addr[dev];
}

mgb_status attention_tc_fwd(const AttnArgs& a, cudaStream_t st);
mgb_status attention_bf16_bwd(const AttnArgs& a, cudaStream_t st);
mgb_status attention_f32_fwd(const AttnArgs& a, cudaStream_t st);
mgb_status attention_f32_bwd(const AttnArgs& a, cudaStream_t st);

mgb_status attention_fwd_launch(const AttnArgs& a, cudaStream_t st) {
  if (a.B == 0 || a.S == 0) return MGB_OK;
  LaunchScope scope(PROF_ATTN_FWD, st, 1);
  return a.dtype == MGB_BF16 ? attention_tc_fwd(a, st) : attention_f32_fwd(a, st);
}
mgb_status attention_bwd_launch(const AttnArgs& a, cudaStream_t st) {
  if (a.B == 0 || a.S == 0) return MGB_OK;
  LaunchScope scope(PROF_ATTN_BWD, st, 3);
  return a.dtype == MGB_BF16 ? attention_bf16_bwd(a, st) : attention_f32_bwd(a, st);
}

bool fault_injected() {
  const char* f = getenv("MGB_FAULT");
  return f != nullptr && strcmp(f, "validate") == 0;
}

mgb_status check_arch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MGB_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MGB_ERR_CUDA;
  return (major == 10 && minor == 3) ? MGB_OK : MGB_ERR_ARCH;
}

namespace {

__global__ void selftest_wait_kernel(unsigned long long limit_ns, int* err) {
  __shared__ uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // nothing ever arrives on this barrier: the bounded wait (the same routine
  // the GEMM pipeline uses) must run out and record the timeout
  if (threadIdx.x == 0) mbar_wait(b, 0, err, limit_ns);
}

#define MGB_TRY(expr)                    \
  do {                                   \
    const mgb_status s_ = (expr);        \
    if (s_ != MGB_OK) return s_;         \
  } while (0)

inline size_t al256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

struct Plan {
  int B, S, T, H, nq, nkv, d, F, W, Wqkv, Dq;
  size_t es;
  bool pre, swiglu;
  // saved buffer
  size_t s_mu1, s_rs1, s_mu2, s_rs2, s_lse, s_xn, s_qkv, s_O, s_h, s_r1, s_hn, s_u, s_a, s_r2;
  size_t s_dmask;  // attention keep bits (attn_dropout > 0)
  size_t saved;
  // backward workspace
  size_t w_dffn, w_dh, w_dr2, w_du, w_dO, w_dqkv, w_dxn, w_delta, w_cparts, w_lparts, w_fparts;
  size_t w_dz1, w_dz2;  // hidden dropout: the projection's / fc2's branch gradients
  size_t w_tf32, tf32_bwd;  // float32: split operands of the three-TF32 GEMMs
  size_t bwd;
  size_t fwd, tf32_fwd;     // forward workspace (float32: the same split scratch)
  int cparts, lparts, fparts;
  bool hdrop;
};

// Dropout of the hidden branch fused into a residual epilogue.
void set_hidden_dropout(const mgb_block_desc* d, const mgb_rng_state& rng, GemmArgs* g) {
  if (!(d->hidden_dropout > 0.0f)) return;
  g->drop_thr = dropout_threshold(d->hidden_dropout);
  g->drop_scale = 256.0f / (float)g->drop_thr;
  g->drop_seed = rng.seed;
  g->drop_offset = rng.offset;
}

// Dropout of the attention probabilities inside the attention kernels; the
// keep bits live in the saved buffer between the forward and the backward.
void set_attn_dropout(const mgb_block_desc* d, const Plan& p, void* saved, AttnArgs* a) {
  if (!(d->attn_dropout > 0.0f)) return;
  a->drop_thr = dropout_threshold(d->attn_dropout);
  a->drop_scale = 256.0f / (float)a->drop_thr;
  a->drop_seed = d->rng_attn.seed;
  a->drop_offset = d->rng_attn.offset;
  a->drop_mask = reinterpret_cast<uint32_t*>(static_cast<char*>(saved) + p.s_dmask);
}

mgb_status validate_desc(const mgb_block_desc* d) {
  if (d == nullptr) return MGB_ERR_INVALID_ARG;
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  if (d->batch < 0 || d->seq < 1 || d->hidden < 1 || d->n_q_heads < 1 || d->n_kv_heads < 1 ||
      d->head_dim < 1 || d->ffn < 1)
    return MGB_ERR_INVALID_ARG;
  if (d->n_q_heads % d->n_kv_heads != 0) return MGB_ERR_INVALID_ARG;
  if (d->dtype != MGB_F32 && d->dtype != MGB_BF16) return MGB_ERR_INVALID_ARG;
  if (d->norm_pos != MGB_PRE_LN && d->norm_pos != MGB_POST_LN) return MGB_ERR_INVALID_ARG;
  if (d->act != MGB_GELU_ERF && d->act != MGB_SWIGLU) return MGB_ERR_INVALID_ARG;
  if (!(d->ln_eps >= 0.0f)) return MGB_ERR_INVALID_ARG;
  if ((d->causal | d->ln_affine | d->has_bias) & ~1) return MGB_ERR_INVALID_ARG;
  const int64_t lim = (int64_t)1 << 31;
  if ((int64_t)d->batch * d->seq >= lim || (int64_t)d->n_q_heads * d->head_dim >= lim)
    return MGB_ERR_INVALID_ARG;
  if (d->act == MGB_SWIGLU) {
    if (d->glu_block < 1 || d->ffn % d->glu_block != 0) return MGB_ERR_INVALID_ARG;
    if (d->dtype == MGB_BF16 && d->glu_block != 32 && d->glu_block != 64 && d->glu_block != 128)
      return MGB_ERR_UNSUPPORTED;
  }
  // every row of every activation / weight a multiple of 16 bytes
  const int vmul = d->dtype == MGB_BF16 ? 8 : 4;
  if (d->hidden % vmul || d->ffn % vmul || (d->n_q_heads * d->head_dim) % vmul ||
      (d->n_kv_heads * d->head_dim) % vmul)
    return MGB_ERR_MISALIGNED;
  if (d->dtype == MGB_BF16 && d->head_dim != 64 && d->head_dim != 128) return MGB_ERR_UNSUPPORTED;
  if (d->dtype == MGB_F32 && (d->head_dim > 256 || d->seq > 2048)) return MGB_ERR_UNSUPPORTED;
  // LayerNorm keeps a row in registers (at most 1024 threads x 4 vectors of 16
  // bytes) and its backward keeps dgamma/dbeta partials of a row in shared memory
  if (d->hidden > 16384) return MGB_ERR_UNSUPPORTED;
  // dropout: probabilities in [0, 1); the hidden sites are fused into the bf16
  // residual epilogues (whole 16-element stream blocks per 32-column chunk)
  // (a probability so close to 1 that no byte is kept is rejected here, before
  // any launch, rather than by a kernel launcher midway through the layer)
  if (!(d->hidden_dropout >= 0.0f && d->hidden_dropout < 1.0f) ||
      !(d->attn_dropout >= 0.0f && d->attn_dropout < 1.0f) ||
      dropout_threshold(d->hidden_dropout) == 0 || dropout_threshold(d->attn_dropout) == 0)
    return MGB_ERR_INVALID_ARG;
  if (d->attn_dropout > 0.0f) {
    // applied in the tcgen05 attention kernels
    if (d->dtype != MGB_BF16) return MGB_ERR_UNSUPPORTED;
    if (d->rng_attn.offset % 16) return MGB_ERR_INVALID_ARG;
  }
  if (d->hidden_dropout > 0.0f) {
    if (d->dtype != MGB_BF16) return MGB_ERR_UNSUPPORTED;
    if (d->hidden % 16 || d->rng_proj.offset % 16 || d->rng_fc2.offset % 16)
      return MGB_ERR_INVALID_ARG;
  }
  return MGB_OK;
}

void make_plan(const mgb_block_desc* d, Plan* p) {
  p->B = d->batch; p->S = d->seq; p->T = d->batch * d->seq;
  p->H = d->hidden; p->nq = d->n_q_heads; p->nkv = d->n_kv_heads; p->d = d->head_dim;
  p->F = d->ffn;
  p->swiglu = d->act == MGB_SWIGLU;
  p->W = p->swiglu ? 2 * d->ffn : d->ffn;
  p->Dq = p->nq * p->d;
  p->Wqkv = (p->nq + 2 * p->nkv) * p->d;
  p->es = d->dtype == MGB_BF16 ? 2 : 4;
  p->pre = d->norm_pos == MGB_PRE_LN;
  const size_t T = p->T, es = p->es;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t at = o; o += al256(bytes); return at; };
  p->s_mu1 = take(4 * T); p->s_rs1 = take(4 * T);
  p->s_mu2 = take(4 * T); p->s_rs2 = take(4 * T);
  p->s_lse = take(4 * (size_t)p->B * p->nq * p->S);
  p->s_xn = p->pre ? take(es * T * p->H) : 0;
  p->s_qkv = take(es * T * p->Wqkv);
  p->s_O = take(es * T * p->Dq);
  p->s_h = take(es * T * p->H);
  p->s_r1 = p->pre ? 0 : take(es * T * p->H);
  p->s_hn = p->pre ? take(es * T * p->H) : 0;
  p->s_u = take(es * T * p->W);
  p->s_a = take(es * T * p->F);
  p->s_r2 = p->pre ? 0 : take(es * T * p->H);
  p->s_dmask = d->attn_dropout > 0.0f ? take(attn_mask_bytes(p->B, p->nq, p->S)) : 0;
  p->saved = o;
  o = 0;
  p->cparts = colsum_parts(p->T);
  p->lparts = layernorm_bwd_parts(p->T);
  const size_t maxN = (size_t)((p->W > p->Wqkv ? p->W : p->Wqkv) > p->H
                                   ? (p->W > p->Wqkv ? p->W : p->Wqkv) : p->H);
  p->w_dffn = take(es * T * p->H);
  p->w_dh = take(es * T * p->H);
  p->w_dr2 = take(es * T * p->H);
  p->w_du = take(es * T * p->W);
  p->w_dO = take(es * T * p->Dq);
  p->w_dqkv = take(es * T * p->Wqkv);
  p->w_dxn = take(es * T * p->H);
  p->w_delta = take(attn_bwd_ws_bytes(p->B, p->S, p->nq));
  p->w_cparts = take(4 * (size_t)p->cparts * maxN);
  p->w_lparts = take(4 * 2 * (size_t)p->lparts * p->H);
  // bf16 with biases: the fc2 input-gradient epilogue leaves db1's partial sums
  // per 32 rows here (the float32 path sums du with the column-sum kernel)
  // (at least one row: with no tokens the reduction zeroes one and sums it)
  p->fparts = (p->T + 31) / 32;
  p->w_fparts = (d->dtype == MGB_BF16 && d->has_bias)
                    ? take(4 * (size_t)(p->fparts > 0 ? p->fparts : 1) * p->W)
                    : 0;
  p->hdrop = d->hidden_dropout > 0.0f;
  p->w_dz1 = p->hdrop ? take(es * T * p->H) : 0;
  p->w_dz2 = p->hdrop ? take(es * T * p->H) : 0;
  // float32: the largest split-operand scratch of the layer's GEMMs (the
  // backward issues its GEMMs in order on one stream, so one region serves)
  p->tf32_fwd = p->tf32_bwd = 0;
  if (d->dtype == MGB_F32) {
    const int Tn = p->T, H = p->H, W = p->W, F = p->F, Dq = p->Dq, Wq = p->Wqkv;
    const int fwd[4][3] = {{Tn, Wq, H}, {Tn, H, Dq}, {Tn, W, H}, {Tn, H, F}};
    const int bwd[8][3] = {{H, F, Tn}, {Tn, F, H}, {W, H, Tn}, {Tn, H, W},
                           {H, Dq, Tn}, {Tn, Dq, H}, {Wq, H, Tn}, {Tn, H, Wq}};
    for (auto& g : fwd) p->tf32_fwd = std::max(p->tf32_fwd, gemm_tf32_scratch_bytes(g[0], g[1], g[2]));
    for (auto& g : bwd) p->tf32_bwd = std::max(p->tf32_bwd, gemm_tf32_scratch_bytes(g[0], g[1], g[2]));
  }
  p->w_tf32 = p->tf32_bwd ? take(p->tf32_bwd) : 0;
  p->bwd = o;
  p->fwd = p->tf32_fwd;
}

mgb_status check_weights(const mgb_block_desc* d, const mgb_block_weights* w) {
  if (w == nullptr) return MGB_ERR_INVALID_ARG;
  if (!w->w_qkv || !w->w_o || !w->w_1 || !w->w_2) return MGB_ERR_INVALID_ARG;
  const bool hb = d->has_bias, ha = d->ln_affine;
  if (hb != (w->b_qkv != nullptr) || hb != (w->b_o != nullptr) || hb != (w->b_1 != nullptr) ||
      hb != (w->b_2 != nullptr))
    return MGB_ERR_INVALID_ARG;
  if (ha != (w->ln1_g != nullptr) || ha != (w->ln1_b != nullptr) || ha != (w->ln2_g != nullptr) ||
      ha != (w->ln2_b != nullptr))
    return MGB_ERR_INVALID_ARG;
  const void* ps[] = {w->w_qkv, w->b_qkv, w->w_o, w->b_o, w->w_1, w->b_1,
                      w->w_2,   w->b_2,   w->ln1_g, w->ln1_b, w->ln2_g, w->ln2_b};
  for (const void* p : ps)
    if (!aligned16(p)) return MGB_ERR_MISALIGNED;
  return MGB_OK;
}

template <typename P>
P* at(void* base, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(base) + off);
}
template <typename P>
const P* at(const void* base, size_t off) {
  return reinterpret_cast<const P*>(static_cast<const char*>(base) + off);
}

GemmArgs mk_gemm(int dtype, int M, int N, int K, int a_mn, const void* A, int64_t lda, int b_mn,
                 const void* B, int64_t ldb, int epi, void* C, int64_t ldc) {
  GemmArgs g;
  g.dtype = dtype; g.M = M; g.N = N; g.K = K;
  g.a_mn = a_mn; g.A = A; g.lda = lda;
  g.b_mn = b_mn; g.B = B; g.ldb = ldb;
  g.epi = epi; g.C = C; g.ldc = ldc;
  return g;
}

}  // namespace
}  // namespace mgb

using namespace mgb;

extern "C" {

int32_t mgb_version(void) { return 100; }

const char* mgb_status_string(mgb_status s) {
  switch (s) {
    case MGB_OK: return "ok";
    case MGB_ERR_INVALID_ARG: return "invalid argument";
    case MGB_ERR_UNSUPPORTED: return "unsupported configuration";
    case MGB_ERR_MISALIGNED: return "pointer or row stride not 16-byte aligned";
    case MGB_ERR_WORKSPACE_TOO_SMALL: return "workspace or saved buffer too small";
    case MGB_ERR_ARCH: return "device is not sm_103 (GB300)";
    case MGB_ERR_CUDA: return "CUDA runtime error";
    case MGB_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case MGB_ERR_NOT_IMPLEMENTED: return "not implemented";
    case MGB_ERR_DEVICE_CHECK: return "a device-side consistency check failed (checking build)";
  }
  return "unknown status";
}

mgb_status mgb_device_status(void* stream) {
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MGB_ERR_CUDA;
  int w = 0;
  if (cudaMemcpyFromSymbol(&w, g_error_word, sizeof(int)) != cudaSuccess) return MGB_ERR_CUDA;
  if (w != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int)) != cudaSuccess) return MGB_ERR_CUDA;
  }
  if (w & kErrTimeout) return MGB_ERR_DEVICE_TIMEOUT;
  return (w & kErrCheck) ? MGB_ERR_DEVICE_CHECK : MGB_OK;
}

mgb_status mgb_memcpy_async(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return MGB_OK;
  if (dst == nullptr || src == nullptr) return MGB_ERR_INVALID_ARG;
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, as_stream(stream)) == cudaSuccess
             ? MGB_OK
             : MGB_ERR_CUDA;
}

mgb_status mgb_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  if (limit_ns > 5000000000ull) return MGB_ERR_INVALID_ARG;
  MGB_TRY(check_arch());
  int* err = device_error_word();
  if (err == nullptr) return MGB_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, as_stream(stream)>>>(limit_ns, err);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

mgb_status mgb_block_sizes(const mgb_block_desc* desc, size_t* saved_bytes, size_t* fwd_ws_bytes,
                           size_t* bwd_ws_bytes) {
  MGB_TRY(validate_desc(desc));
  Plan p;
  make_plan(desc, &p);
  if (saved_bytes) *saved_bytes = p.saved;
  if (fwd_ws_bytes) *fwd_ws_bytes = p.fwd;
  if (bwd_ws_bytes) *bwd_ws_bytes = p.bwd;
  return MGB_OK;
}

mgb_status mgb_block_fwd(const mgb_block_desc* desc, const mgb_block_weights* w, const void* x,
                         void* y, void* saved, size_t saved_bytes, void* ws, size_t ws_bytes,
                         void* stream) {
  MGB_TRY(validate_desc(desc));
  MGB_TRY(check_weights(desc, w));
  Plan p;
  make_plan(desc, &p);
  if (!x || !y || !saved || (p.fwd > 0 && !ws)) return MGB_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(saved)) return MGB_ERR_MISALIGNED;
  if (ws && (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MGB_ERR_MISALIGNED;
  if (saved_bytes < p.saved || ws_bytes < p.fwd) return MGB_ERR_WORKSPACE_TOO_SMALL;
  MGB_TRY(check_arch());
  if (p.T == 0) return MGB_OK;
  cudaStream_t st = as_stream(stream);
  const int dt = desc->dtype;
  const int T = p.T, H = p.H;
  // float32: every GEMM runs as three TF32 products with its split operands in ws
  auto scr = [&](GemmArgs g) {
    if (dt == MGB_F32) { g.scratch = ws; g.scratch_bytes = p.fwd; }
    return g;
  };
  float* mu1 = at<float>(saved, p.s_mu1); float* rs1 = at<float>(saved, p.s_rs1);
  float* mu2 = at<float>(saved, p.s_mu2); float* rs2 = at<float>(saved, p.s_rs2);
  float* lse = at<float>(saved, p.s_lse);
  void* qkv = at<char>(saved, p.s_qkv);
  void* O = at<char>(saved, p.s_O);
  void* h = at<char>(saved, p.s_h);
  void* u = at<char>(saved, p.s_u);
  void* a = at<char>(saved, p.s_a);

  // attention sublayer input
  std::unique_ptr<LaunchScope> stage(new LaunchScope(PROF_STAGE_ATTN, st, 1, false));
  const void* a_in = x;
  if (p.pre) {
    void* xn = at<char>(saved, p.s_xn);
    MGB_TRY(layernorm_fwd_launch(T, H, dt, desc->ln_eps, x, w->ln1_g, w->ln1_b, xn, mu1, rs1, st));
    a_in = xn;
  }
  GemmArgs g = mk_gemm(dt, T, p.Wqkv, H, 0, a_in, H, 0, w->w_qkv, H, EPI_STORE, qkv, p.Wqkv);
  g.bias = w->b_qkv;
  MGB_TRY(gemm_launch(scr(g), st));

  AttnArgs at_{};
  at_.B = p.B; at_.S = p.S; at_.nq = p.nq; at_.nkv = p.nkv; at_.d = p.d;
  at_.causal = desc->causal; at_.dtype = dt;
  at_.q = qkv;
  at_.k = static_cast<char*>(qkv) + p.es * p.Dq;
  at_.v = static_cast<char*>(qkv) + p.es * (p.Dq + (size_t)p.nkv * p.d);
  at_.ld_q = p.Wqkv; at_.ld_kv = p.Wqkv;
  at_.o = O; at_.ld_o = p.Dq; at_.lse = lse;
  set_attn_dropout(desc, p, saved, &at_);
  MGB_TRY(attention_fwd_launch(at_, st));

  // output projection + residual (Pre: h; Post: r1 then h = LN1(r1))
  void* r1 = p.pre ? h : at<char>(saved, p.s_r1);
  g = mk_gemm(dt, T, H, p.Dq, 0, O, p.Dq, 0, w->w_o, p.Dq, EPI_BIAS_RESID, r1, H);
  g.bias = w->b_o; g.resid = x; g.ldr = H;
  set_hidden_dropout(desc, desc->rng_proj, &g);
  MGB_TRY(gemm_launch(scr(g), st));
  const void* f_in;
  if (!p.pre)
    MGB_TRY(layernorm_fwd_launch(T, H, dt, desc->ln_eps, r1, w->ln1_g, w->ln1_b, h, mu1, rs1, st));
  stage.reset(new LaunchScope(PROF_STAGE_FFN, st, 1, false));
  if (p.pre) {
    void* hn = at<char>(saved, p.s_hn);
    MGB_TRY(layernorm_fwd_launch(T, H, dt, desc->ln_eps, h, w->ln2_g, w->ln2_b, hn, mu2, rs2, st));
    f_in = hn;
  } else {
    f_in = h;
  }
  // fc1 + activation
  g = mk_gemm(dt, T, p.W, H, 0, f_in, H, 0, w->w_1, H,
              p.swiglu ? EPI_BIAS_SWIGLU : EPI_BIAS_GELU, u, p.W);
  g.bias = w->b_1; g.C2 = a; g.ldc2 = p.F; g.glu_block = desc->glu_block;
  MGB_TRY(gemm_launch(scr(g), st));
  // fc2 + residual (Pre: y; Post: r2 then y = LN2(r2))
  void* r2 = p.pre ? y : at<char>(saved, p.s_r2);
  g = mk_gemm(dt, T, H, p.F, 0, a, p.F, 0, w->w_2, p.F, EPI_BIAS_RESID, r2, H);
  g.bias = w->b_2; g.resid = h; g.ldr = H;
  set_hidden_dropout(desc, desc->rng_fc2, &g);
  MGB_TRY(gemm_launch(scr(g), st));
  if (!p.pre)
    MGB_TRY(layernorm_fwd_launch(T, H, dt, desc->ln_eps, r2, w->ln2_g, w->ln2_b, y, mu2, rs2, st));
  return MGB_OK;
}

mgb_status mgb_block_bwd(const mgb_block_desc* desc, const mgb_block_weights* w, const void* x,
                         const void* dy, const void* saved, size_t saved_bytes, void* dx,
                         const mgb_block_grads* gr, void* ws, size_t ws_bytes, void* stream) {
  MGB_TRY(validate_desc(desc));
  MGB_TRY(check_weights(desc, w));
  Plan p;
  make_plan(desc, &p);
  if (!x || !dy || !saved || !dx || !gr || (!ws && p.bwd > 0)) return MGB_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(dy) || !aligned16(saved) || !aligned16(dx) || !aligned16(ws))
    return MGB_ERR_MISALIGNED;
  {
    const void* gs[] = {gr->w_qkv, gr->b_qkv, gr->w_o, gr->b_o, gr->w_1, gr->b_1,
                        gr->w_2,   gr->b_2,   gr->ln1_g, gr->ln1_b, gr->ln2_g, gr->ln2_b};
    for (const void* q : gs)
      if (!aligned16(q)) return MGB_ERR_MISALIGNED;
    if (!desc->has_bias && (gr->b_qkv || gr->b_o || gr->b_1 || gr->b_2)) return MGB_ERR_INVALID_ARG;
    if (!desc->ln_affine && (gr->ln1_g || gr->ln1_b || gr->ln2_g || gr->ln2_b))
      return MGB_ERR_INVALID_ARG;
  }
  if (saved_bytes < p.saved) return MGB_ERR_WORKSPACE_TOO_SMALL;
  if (ws_bytes < p.bwd) return MGB_ERR_WORKSPACE_TOO_SMALL;
  MGB_TRY(check_arch());
  cudaStream_t st = as_stream(stream);
  // ends (destroyed last) after the side streams are joined back
  LaunchScope stage(PROF_STAGE_BWD, st, 1, false);
  const int dt = desc->dtype;
  const int T = p.T, H = p.H;
  // float32: every GEMM runs as three TF32 products with its split operands in
  // the workspace, in order on one stream (one scratch region)
  auto scr = [&](GemmArgs g) {
    if (dt == MGB_F32) { g.scratch = at<char>(ws, p.w_tf32); g.scratch_bytes = p.tf32_bwd; }
    return g;
  };
  const float* mu1 = at<float>(saved, p.s_mu1); const float* rs1 = at<float>(saved, p.s_rs1);
  const float* mu2 = at<float>(saved, p.s_mu2); const float* rs2 = at<float>(saved, p.s_rs2);
  const float* lse = at<float>(saved, p.s_lse);
  const void* qkv = at<char>(saved, p.s_qkv);
  const void* O = at<char>(saved, p.s_O);
  const void* h = at<char>(saved, p.s_h);
  const void* u = at<char>(saved, p.s_u);
  const void* a = at<char>(saved, p.s_a);
  const void* a_in = p.pre ? at<char>(saved, p.s_xn) : x;
  const void* f_in = p.pre ? at<char>(saved, p.s_hn) : h;
  void* d_ffn = at<char>(ws, p.w_dffn);
  void* d_h = at<char>(ws, p.w_dh);
  void* d_r2 = at<char>(ws, p.w_dr2);
  void* du = at<char>(ws, p.w_du);
  void* dO = at<char>(ws, p.w_dO);
  void* dqkv = at<char>(ws, p.w_dqkv);
  void* dxn = at<char>(ws, p.w_dxn);
  float* delta = at<float>(ws, p.w_delta);
  float* cparts = at<float>(ws, p.w_cparts);
  float* lparts = at<float>(ws, p.w_lparts);

  // The input-gradient chain (dgrad GEMMs, LayerNorm and attention backward)
  // runs on the caller's stream; each weight gradient and bias column sum is
  // issued on the side stream once its inputs exist there. Only the side
  // stream uses cparts; only the caller's stream uses lparts.
  SideLane lane(st, nullptr, 0, dt == MGB_F32);
  cudaStream_t s2 = lane.side();
  // gradient at the fc2 residual sum (Pre: dy itself; Post: through LN2)
  const void* dr2 = dy;
  if (!p.pre) {
    MGB_TRY(layernorm_bwd_launch(T, H, dt, at<char>(saved, p.s_r2), mu2, rs2, w->ln2_g, dy, nullptr,
                                 d_r2, gr->ln2_g, gr->ln2_b, lparts, p.lparts, st));
    dr2 = d_r2;
  }
  // through the hidden dropout of fc2's branch (the residual path keeps dr2)
  const void* dz2 = dr2;
  if (p.hdrop) {
    MGB_TRY(dropout_launch(T, H, dt, desc->hidden_dropout, desc->rng_fc2.seed, desc->rng_fc2.offset,
                           dr2, H, at<char>(ws, p.w_dz2), H, st));
    dz2 = at<char>(ws, p.w_dz2);
  }
  // fc2: db2, dW2 = dz2^T a, du = (dz2 W2) * act'(u)
  MGB_TRY(lane.fork());
  if (gr->b_2) MGB_TRY(colsum_launch(T, H, dt, dz2, H, gr->b_2, cparts, p.cparts, s2));
  if (gr->w_2)
    MGB_TRY(gemm_launch(scr(mk_gemm(dt, H, p.F, T, 1, dz2, H, 1, a, p.F, EPI_STORE, gr->w_2, p.F)), s2));
  const bool fused_db1 = gr->b_1 != nullptr && dt == MGB_BF16;
  {
    GemmArgs g = mk_gemm(dt, T, p.F, H, 0, dz2, H, 1, w->w_2, p.F,
                         p.swiglu ? EPI_DSWIGLU : EPI_DGELU, du, p.W);
    g.aux = u; g.ldaux = p.W; g.glu_block = desc->glu_block;
    if (fused_db1) g.colsum_part = at<float>(ws, p.w_fparts);
    MGB_TRY(gemm_launch(scr(g), st));
  }
  // fc1: db1 (from the partials of the epilogue above, or a column sum of du),
  // dW1 = du^T f_in, d f_in = du W1
  MGB_TRY(lane.fork());
  if (fused_db1)
    MGB_TRY(colsum_reduce_launch(T > 0 ? p.fparts : 0, p.W, dt, at<float>(ws, p.w_fparts),
                                 gr->b_1, s2));
  if (gr->b_1 && !fused_db1)
    MGB_TRY(colsum_launch(T, p.W, dt, du, p.W, gr->b_1, cparts, p.cparts, s2));
  if (gr->w_1)
    MGB_TRY(gemm_launch(scr(mk_gemm(dt, p.W, H, T, 1, du, p.W, 1, f_in, H, EPI_STORE, gr->w_1, H)), s2));
  const void* dr1;
  if (p.pre) {
    MGB_TRY(gemm_launch(scr(mk_gemm(dt, T, H, p.W, 0, du, p.W, 1, w->w_1, H, EPI_STORE, d_ffn, H)), st));
    // dh = dy + LN2_bwd(d hn)
    MGB_TRY(layernorm_bwd_launch(T, H, dt, h, mu2, rs2, w->ln2_g, d_ffn, dy, d_h, gr->ln2_g,
                                 gr->ln2_b, lparts, p.lparts, st));
    dr1 = d_h;
  } else {
    // dh = du W1 + dr2 (h feeds fc1 and the fc2 residual), dr1 = LN1_bwd(dh)
    GemmArgs g = mk_gemm(dt, T, H, p.W, 0, du, p.W, 1, w->w_1, H, EPI_BIAS_RESID, d_h, H);
    g.resid = dr2; g.ldr = H;
    MGB_TRY(gemm_launch(scr(g), st));
    MGB_TRY(layernorm_bwd_launch(T, H, dt, at<char>(saved, p.s_r1), mu1, rs1, w->ln1_g, d_h,
                                 nullptr, d_ffn, gr->ln1_g, gr->ln1_b, lparts, p.lparts, st));
    dr1 = d_ffn;
  }
  // through the hidden dropout of the projection's branch
  const void* dz1 = dr1;
  if (p.hdrop) {
    MGB_TRY(dropout_launch(T, H, dt, desc->hidden_dropout, desc->rng_proj.seed,
                           desc->rng_proj.offset, dr1, H, at<char>(ws, p.w_dz1), H, st));
    dz1 = at<char>(ws, p.w_dz1);
  }
  // output projection: dbo, dWo = dz1^T O, dO = dz1 Wo
  MGB_TRY(lane.fork());
  if (gr->b_o) MGB_TRY(colsum_launch(T, H, dt, dz1, H, gr->b_o, cparts, p.cparts, s2));
  if (gr->w_o)
    MGB_TRY(gemm_launch(scr(mk_gemm(dt, H, p.Dq, T, 1, dz1, H, 1, O, p.Dq, EPI_STORE, gr->w_o, p.Dq)), s2));
  MGB_TRY(gemm_launch(scr(mk_gemm(dt, T, p.Dq, H, 0, dz1, H, 1, w->w_o, p.Dq, EPI_STORE, dO, p.Dq)), st));
  // attention backward into the fused dqkv buffer
  {
    AttnArgs at_{};
    at_.B = p.B; at_.S = p.S; at_.nq = p.nq; at_.nkv = p.nkv; at_.d = p.d;
    at_.causal = desc->causal; at_.dtype = dt;
    at_.q = qkv;
    at_.k = static_cast<const char*>(qkv) + p.es * p.Dq;
    at_.v = static_cast<const char*>(qkv) + p.es * (p.Dq + (size_t)p.nkv * p.d);
    at_.ld_q = p.Wqkv; at_.ld_kv = p.Wqkv;
    at_.o = const_cast<void*>(O); at_.ld_o = p.Dq; at_.lse = const_cast<float*>(lse);
    at_.dout = dO; at_.ld_do = p.Dq;
    at_.dq = dqkv;
    at_.dk = static_cast<char*>(dqkv) + p.es * p.Dq;
    at_.dv = static_cast<char*>(dqkv) + p.es * (p.Dq + (size_t)p.nkv * p.d);
    at_.ld_dq = p.Wqkv; at_.ld_dkv = p.Wqkv;
    at_.delta = delta;
    set_attn_dropout(desc, p, const_cast<void*>(saved), &at_);
    MGB_TRY(attention_bwd_launch(at_, st));
  }
  // QKV: dbqkv, dWqkv = dqkv^T a_in, d a_in = dqkv Wqkv
  MGB_TRY(lane.fork());
  if (gr->b_qkv) MGB_TRY(colsum_launch(T, p.Wqkv, dt, dqkv, p.Wqkv, gr->b_qkv, cparts, p.cparts, s2));
  if (gr->w_qkv)
    MGB_TRY(gemm_launch(
        scr(mk_gemm(dt, p.Wqkv, H, T, 1, dqkv, p.Wqkv, 1, a_in, H, EPI_STORE, gr->w_qkv, H)), s2));
  if (p.pre) {
    MGB_TRY(gemm_launch(scr(mk_gemm(dt, T, H, p.Wqkv, 0, dqkv, p.Wqkv, 1, w->w_qkv, H, EPI_STORE, dxn, H)),
                        st));
    MGB_TRY(layernorm_bwd_launch(T, H, dt, x, mu1, rs1, w->ln1_g, dxn, dr1, dx, gr->ln1_g, gr->ln1_b,
                                 lparts, p.lparts, st));
  } else {
    GemmArgs g = mk_gemm(dt, T, H, p.Wqkv, 0, dqkv, p.Wqkv, 1, w->w_qkv, H, EPI_BIAS_RESID, dx, H);
    g.resid = dr1; g.ldr = H;
    MGB_TRY(gemm_launch(scr(g), st));
  }
  return lane.join();
}

// ------------------------------------------------------------ cross-entropy

static mgb_status validate_ce(const mgb_ce_desc* d) {
  if (d == nullptr) return MGB_ERR_INVALID_ARG;
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  if (d->tokens < 0 || d->hidden < 1 || d->vocab < 1 || d->chunk < 1) return MGB_ERR_INVALID_ARG;
  if (d->dtype != MGB_BF16) return MGB_ERR_UNSUPPORTED;
  if (d->hidden % 8 || d->vocab % 8 || d->chunk % 8) return MGB_ERR_MISALIGNED;
  if (!(d->grad_scale == d->grad_scale)) return MGB_ERR_INVALID_ARG;
  if (d->mode != MGB_CE_STREAM && d->mode != MGB_CE_FUSED && d->mode != MGB_CE_RESIDENT &&
      d->mode != MGB_CE_BLOCKED)
    return MGB_ERR_INVALID_ARG;
  if (d->token_block < 0) return MGB_ERR_INVALID_ARG;
  return MGB_OK;
}

struct CEPlan {
  int n_chunks, C, n_parts, n_t;
  size_t logits, m, s, t, lse, dh, bl, split, total;
  // MGB_CE_BLOCKED: rows per token block, blocks, K ranges of the d_hidden
  // product and their partial planes, the float32 d_emb accumulator
  int tb, n_blocks, dh_splits;
  size_t dh_part, de_acc;
};

constexpr int kCeDefaultTokenBlock = 4096;

// K ranges (whole 64-wide blocks) of the split-K GEMM for a request of
// `want` ranges, as the kernel cuts them.
static int splitk_ranges(int K, int want) {
  const int num_k = (K + 63) / 64;
  if (want <= 1 || num_k <= 1) return 1;
  const int per = (num_k + want - 1) / want;
  return (num_k + per - 1) / per;
}

// Partials: one per chunk (streaming) or one per chunk and 128-column group
// (fused, written by the GEMM epilogue); target logits per chunk (streaming,
// zero outside the chunk) or one array each token's owning tile writes (fused).
static void ce_plan(const mgb_ce_desc* d, CEPlan* p) {
  size_t T = d->tokens;
  p->C = d->chunk < d->vocab ? d->chunk : d->vocab;
  p->n_chunks = (d->vocab + p->C - 1) / p->C;
  const bool resident = d->mode == MGB_CE_RESIDENT;
  const bool blocked = d->mode == MGB_CE_BLOCKED;
  const bool fused = d->mode == MGB_CE_FUSED || resident || blocked;
  p->tb = 0;
  p->n_blocks = 0;
  p->dh_splits = 1;
  p->dh_part = p->de_acc = 0;
  const size_t T_all = T;
  if (blocked) {
    // rows per block: a multiple of 256 (the combine's block sums then fall
    // on the same 256-token groups as a single combine over all tokens)
    int tb = d->token_block > 0 ? d->token_block : kCeDefaultTokenBlock;
    tb = (tb + 255) / 256 * 256;
    const int t_all = (d->tokens + 255) / 256 * 256;
    p->tb = tb < t_all ? tb : (t_all > 0 ? t_all : 256);
    p->n_blocks = (d->tokens + p->tb - 1) / p->tb;
    p->dh_splits = splitk_ranges(d->vocab, gemm_splitk_count(p->tb, d->hidden, d->vocab, 16));
    T = p->tb;  // the per-block planes below are sized for one block
  }
  p->n_parts = 0;
  for (int c = 0; c < p->n_chunks; ++c) {
    const int v0 = c * p->C, Cc = (d->vocab - v0) < p->C ? (d->vocab - v0) : p->C;
    p->n_parts += fused ? (Cc + 127) / 128 : 1;
  }
  p->n_t = fused ? 1 : p->n_chunks;
  size_t o = 0;
  auto take = [&](size_t bytes) { const size_t a = o; o += al256(bytes); return a; };
  p->logits = take(2 * T * ((resident || blocked) ? (size_t)d->vocab : (size_t)p->C));
  p->m = take(4 * T * p->n_parts);
  p->s = take(4 * T * p->n_parts);
  p->t = take(4 * T * p->n_t);
  p->lse = take(4 * T_all);
  p->dh = (resident || blocked) ? 0 : take(4 * T * d->hidden);
  p->bl = take(4 * (size_t)ce_combine_blocks((int)T_all));
  p->split = p->n_parts > kCeSplits ? take(4 * 2 * (size_t)kCeSplits * T) : 0;
  if (blocked) {
    p->dh_part = take(4 * (size_t)p->dh_splits * T * d->hidden);
    p->de_acc = p->n_blocks > 1 ? take(4 * (size_t)d->vocab * d->hidden) : 0;
  }
  p->total = o;
}

// MGB_CE_BLOCKED: per block of tokens, the logits of every vocab chunk with
// their partials, the block's LSE and losses, G in place, then d_hidden rows
// (split-K) beside d_emb += G^T hidden on the side stream.
static mgb_status ce_blocked(const mgb_ce_desc* desc, const CEPlan& p, const void* hidden,
                             const bf16* E, const int32_t* targets, float* loss_per_token,
                             float* loss_mean, float* lse_buf, void* d_hidden, void* d_emb,
                             void* ws, cudaStream_t st) {
  const int T = desc->tokens, H = desc->hidden, V = desc->vocab, C = p.C;
  bf16* logits = at<bf16>(ws, p.logits);
  float* m = at<float>(ws, p.m);
  float* s = at<float>(ws, p.s);
  float* t = at<float>(ws, p.t);
  float* bl = at<float>(ws, p.bl);
  float* split = p.n_parts > kCeSplits ? at<float>(ws, p.split) : nullptr;
  float* dh_part = at<float>(ws, p.dh_part);
  float* de_acc = at<float>(ws, p.de_acc);
  const bf16* hid = static_cast<const bf16*>(hidden);
  const bool grads = d_hidden || d_emb;
  for (int b = 0; b < p.n_blocks; ++b) {
    const int r0 = b * p.tb;
    const int rows = (T - r0) < p.tb ? (T - r0) : p.tb;
    const bool last = b == p.n_blocks - 1;
    // ---- forward of the block: partials per chunk and 128-column group
    if (cudaMemsetAsync(t, 0, sizeof(float) * rows, st) != cudaSuccess) return MGB_ERR_CUDA;
    {
      // every vocab chunk in one launch (tiles never straddle two chunks):
      // chunk c's partials are planes c * ceil(C / 128) .. of m and s
      GemmArgs g = mk_gemm(MGB_BF16, rows, V, H, 0, hid + (size_t)r0 * H, H, 0, E, H,
                           EPI_CE_STATS, m, 8);
      g.C2 = s; g.ldc2 = 8;
      g.n_chunk = C;
      g.tgt = targets + r0; g.tgt_v0 = 0; g.tgt_out = t;
      if (grads) { g.keep = logits; g.ld_keep = V; }
      g.prof_kind = PROF_GEMM_CE_LOGITS;
      MGB_TRY(gemm_launch(g, st));
    }
    MGB_TRY(ce_combine_launch(rows, p.n_parts, m, s, 1, t, lse_buf + r0, loss_per_token + r0,
                              nullptr, bl + r0 / 256, split, st));
    if (!grads) continue;
    // ---- backward of the block: G in place, then its two products
    MGB_TRY(ce_grad_launch(rows, V, 0, logits, V, targets + r0, lse_buf + r0, desc->grad_scale,
                           st));
    // (destroyed after the lane below: ends once the side stream is joined)
    LaunchScope products(PROF_STAGE_CE_PRODUCTS, st, 1, false);
    SideLane lane(st, last ? as_stream(desc->emb_stream) : nullptr);
    if (d_emb) {
      MGB_TRY(lane.fork());
      GemmArgs g;
      if (p.n_blocks == 1) {
        g = mk_gemm(MGB_BF16, V, H, rows, 1, logits, V, 1, hid + (size_t)r0 * H, H, EPI_STORE,
                    d_emb, H);
      } else {
        // float32 accumulator across blocks: the first block stores its
        // product, the others reduce-add theirs in L2 (TMA bulk copies)
        g = mk_gemm(MGB_BF16, V, H, rows, 1, logits, V, 1, hid + (size_t)r0 * H, H, EPI_F32,
                    de_acc, H);
        g.accumulate = b > 0;
        g.f32_tma = 1;
      }
      g.prof_kind = PROF_GEMM_CE_WGRAD;
      MGB_TRY(gemm_launch(g, lane.side()));
      if (last && p.n_blocks > 1)  // d_emb = bf16(accumulator)
        MGB_TRY(splitk_reduce_launch(V, H, 1, de_acc, 0, H, d_emb, H, lane.side()));
    }
    if (d_hidden) {
      GemmArgs g = mk_gemm(MGB_BF16, rows, H, V, 0, logits, V, 1, E, H, EPI_F32, dh_part, H);
      g.k_splits = p.dh_splits;
      g.split_stride = (int64_t)rows * H;
      g.prof_kind = PROF_GEMM_CE_DGRAD;
      MGB_TRY(gemm_launch(g, st));
      MGB_TRY(splitk_reduce_launch(rows, H, p.dh_splits, dh_part, (int64_t)rows * H, H,
                                   static_cast<bf16*>(d_hidden) + (size_t)r0 * H, H, st));
    }
    MGB_TRY(lane.join());  // the next block overwrites the logits
  }
  return ce_mean_launch(ce_combine_blocks(T), T, bl, loss_mean, st);
}

mgb_status mgb_vocab_ce_sizes(const mgb_ce_desc* desc, size_t* ws_bytes) {
  MGB_TRY(validate_ce(desc));
  CEPlan p;
  ce_plan(desc, &p);
  if (ws_bytes) *ws_bytes = p.total;
  return MGB_OK;
}

mgb_status mgb_vocab_ce_fwd_bwd(const mgb_ce_desc* desc, const void* hidden, const void* emb,
                                const int32_t* targets, float* loss_per_token, float* loss_mean,
                                float* lse, void* d_hidden, void* d_emb, void* ws, size_t ws_bytes,
                                void* stream) {
  MGB_TRY(validate_ce(desc));
  CEPlan p;
  ce_plan(desc, &p);
  if (!hidden || !emb || !targets || !loss_per_token || !loss_mean || !ws)
    return MGB_ERR_INVALID_ARG;
  const void* ptrs[] = {hidden, emb, targets, loss_per_token, lse, d_hidden, d_emb, ws};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MGB_ERR_MISALIGNED;
  if (ws_bytes < p.total) return MGB_ERR_WORKSPACE_TOO_SMALL;
  MGB_TRY(check_arch());
  cudaStream_t st = as_stream(stream);
  const int T = desc->tokens, H = desc->hidden, V = desc->vocab, C = p.C;
  void* logits = at<char>(ws, p.logits);
  float* m = at<float>(ws, p.m);
  float* s = at<float>(ws, p.s);
  float* t = at<float>(ws, p.t);
  float* lse_buf = lse ? lse : at<float>(ws, p.lse);
  float* dh_acc = at<float>(ws, p.dh);
  float* bl = at<float>(ws, p.bl);
  const bf16* E = static_cast<const bf16*>(emb);
  MGB_TRY(ce_check_targets_launch(T, V, targets, st));
  if (desc->mode == MGB_CE_BLOCKED)
    return ce_blocked(desc, p, hidden, E, targets, loss_per_token, loss_mean, lse_buf, d_hidden,
                      d_emb, ws, st);
  const bool resident = desc->mode == MGB_CE_RESIDENT;
  const bool fused = desc->mode == MGB_CE_FUSED || resident;
  // ---- forward: per-chunk partials, then the combine
  if (fused && T > 0 && cudaMemsetAsync(t, 0, sizeof(float) * T, st) != cudaSuccess)
    return MGB_ERR_CUDA;
  for (int c = 0, part = 0; c < p.n_chunks; ++c) {
    const int v0 = c * C, Cc = (V - v0) < C ? (V - v0) : C;
    if (fused) {
      // (max, sum exp) per token and 128 columns straight from the accumulator
      GemmArgs g = mk_gemm(MGB_BF16, T, Cc, H, 0, hidden, H, 0, E + (size_t)v0 * H, H,
                           EPI_CE_STATS, m + (size_t)part * T, 8);
      g.C2 = s + (size_t)part * T; g.ldc2 = 8;
      g.tgt = targets; g.tgt_v0 = v0; g.tgt_out = t;
      if (resident) { g.keep = static_cast<bf16*>(logits) + v0; g.ld_keep = V; }
      g.prof_kind = PROF_GEMM_CE_LOGITS;
      MGB_TRY(gemm_launch(g, st));
      part += (Cc + 127) / 128;
    } else {
      GemmArgs g = mk_gemm(MGB_BF16, T, Cc, H, 0, hidden, H, 0, E + (size_t)v0 * H, H, EPI_STORE,
                           logits, C);
      // the target logit is taken in float32 from the accumulator, not from
      // the bf16 logits the streaming pass reads
      g.tgt = targets; g.tgt_v0 = v0; g.tgt_out = t + (size_t)c * T;
      g.prof_kind = PROF_GEMM_CE_LOGITS;
      MGB_TRY(gemm_launch(g, st));
      MGB_TRY(ce_stats_launch(T, Cc, v0, logits, C, targets, m + (size_t)c * T, s + (size_t)c * T,
                              t + (size_t)c * T, st));
    }
  }
  MGB_TRY(ce_combine_launch(T, p.n_parts, m, s, p.n_t, t, lse_buf, loss_per_token, loss_mean, bl,
                            p.n_parts > kCeSplits ? at<float>(ws, p.split) : nullptr, st));
  if (!d_hidden && !d_emb) return MGB_OK;
  if (resident) {
    // ---- backward over the resident logits: G in place, then
    // d_hidden = G E on this stream and d_emb = G^T hidden on the side stream
    MGB_TRY(ce_grad_launch(T, V, 0, logits, V, targets, lse_buf, desc->grad_scale, st));
    SideLane lane(st, as_stream(desc->emb_stream));
    if (d_emb) {
      MGB_TRY(lane.fork());
      GemmArgs g = mk_gemm(MGB_BF16, V, H, T, 1, logits, V, 1, hidden, H, EPI_STORE, d_emb, H);
      g.prof_kind = PROF_GEMM_CE_WGRAD;
      MGB_TRY(gemm_launch(g, lane.side()));
    }
    if (d_hidden) {
      GemmArgs g = mk_gemm(MGB_BF16, T, H, V, 0, logits, V, 1, E, H, EPI_STORE, d_hidden, H);
      g.prof_kind = PROF_GEMM_CE_DGRAD;
      MGB_TRY(gemm_launch(g, st));
    }
    return lane.join();
  }
  // ---- backward: per chunk, G then its two GEMMs
  for (int c = 0; c < p.n_chunks; ++c) {
    const int v0 = c * C, Cc = (V - v0) < C ? (V - v0) : C;
    if (fused) {
      GemmArgs g = mk_gemm(MGB_BF16, T, Cc, H, 0, hidden, H, 0, E + (size_t)v0 * H, H,
                           EPI_CE_GRAD, logits, C);
      g.tgt = targets; g.tgt_v0 = v0; g.ce_lse = lse_buf; g.ce_scale = desc->grad_scale;
      g.prof_kind = PROF_GEMM_CE_LOGITS;
      MGB_TRY(gemm_launch(g, st));
    } else {
      GemmArgs g = mk_gemm(MGB_BF16, T, Cc, H, 0, hidden, H, 0, E + (size_t)v0 * H, H, EPI_STORE,
                           logits, C);
      g.prof_kind = PROF_GEMM_CE_LOGITS;
      MGB_TRY(gemm_launch(g, st));
      MGB_TRY(ce_grad_launch(T, Cc, v0, logits, C, targets, lse_buf, desc->grad_scale, st));
    }
    if (d_hidden) {
      GemmArgs g = mk_gemm(MGB_BF16, T, H, Cc, 0, logits, C, 1, E + (size_t)v0 * H, H, EPI_F32,
                           dh_acc, H);
      g.accumulate = c > 0;
      if (c == p.n_chunks - 1) { g.C2 = d_hidden; g.ldc2 = H; }
      g.prof_kind = PROF_GEMM_CE_DGRAD;
      MGB_TRY(gemm_launch(g, st));
    }
    if (d_emb) {
      GemmArgs g = mk_gemm(MGB_BF16, Cc, H, T, 1, logits, C, 1, hidden, H, EPI_STORE,
                           static_cast<bf16*>(d_emb) + (size_t)v0 * H, H);
      g.prof_kind = PROF_GEMM_CE_WGRAD;
      MGB_TRY(gemm_launch(g, st));
    }
  }
  return MGB_OK;
}

// ------------------------------------------------------------ building blocks

mgb_status mgb_gemm(const mgb_gemm_desc* d, const void* a, const void* b, const void* bias, void* c,
                    void* stream) {
  if (d == nullptr) return MGB_ERR_INVALID_ARG;
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  GemmArgs g = mk_gemm(d->dtype, d->m, d->n, d->k, d->a_major, a, d->lda, d->b_major, b, d->ldb,
                       (d->c_f32 || d->dtype == MGB_F32) ? EPI_F32 : EPI_STORE, c, d->ldc);
  if ((d->a_major | d->b_major) & ~1) return MGB_ERR_INVALID_ARG;
  if (d->accumulate && !(d->c_f32 || d->dtype == MGB_F32)) return MGB_ERR_INVALID_ARG;
  g.bias = bias;
  g.alpha = d->alpha;
  g.accumulate = d->accumulate;
  MGB_TRY(gemm_check(g));
  MGB_TRY(check_arch());
  return gemm_launch(g, as_stream(stream));
}

mgb_status mgb_gemm_ex(const mgb_gemm_ex_desc* e, const void* a, const void* b, const void* bias,
                       void* c, void* c2, const void* resid, const void* aux, void* stream) {
  if (e == nullptr) return MGB_ERR_INVALID_ARG;
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  const mgb_gemm_desc* d = &e->g;
  if (e->epilogue < MGB_EPI_STORE || e->epilogue > MGB_EPI_F32) return MGB_ERR_INVALID_ARG;
  if ((d->a_major | d->b_major) & ~1) return MGB_ERR_INVALID_ARG;
  // the public values are the library's own epilogue codes
  static_assert((int)MGB_EPI_BIAS_SWIGLU == (int)EPI_BIAS_SWIGLU && (int)MGB_EPI_F32 == (int)EPI_F32,
                "epilogue codes");
  if (d->accumulate && e->epilogue != MGB_EPI_F32) return MGB_ERR_INVALID_ARG;
  GemmArgs g = mk_gemm(d->dtype, d->m, d->n, d->k, d->a_major, a, d->lda, d->b_major, b, d->ldb,
                       e->epilogue, c, d->ldc);
  g.bias = bias;
  g.alpha = d->alpha;
  g.accumulate = d->accumulate;
  g.C2 = c2; g.ldc2 = e->ldc2;
  g.resid = resid; g.ldr = e->ldr;
  g.aux = aux; g.ldaux = e->ldaux;
  g.glu_block = e->glu_block;
  MGB_TRY(gemm_check(g));
  MGB_TRY(check_arch());
  return gemm_launch(g, as_stream(stream));
}

size_t mgb_gemm_f32_tc_ws_bytes(int32_t m, int32_t n, int32_t k) {
  return gemm_tf32_scratch_bytes(m, n, k);
}

mgb_status mgb_gemm_f32_tc(const mgb_gemm_ex_desc* e, const void* a, const void* b,
                           const void* bias, void* c, void* c2, const void* resid, const void* aux,
                           void* ws, size_t ws_bytes, void* stream) {
  if (e == nullptr) return MGB_ERR_INVALID_ARG;
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  const mgb_gemm_desc* d = &e->g;
  if (d->dtype != MGB_F32) return MGB_ERR_INVALID_ARG;
  if (e->epilogue < MGB_EPI_STORE || e->epilogue > MGB_EPI_F32) return MGB_ERR_INVALID_ARG;
  if ((d->a_major | d->b_major) & ~1) return MGB_ERR_INVALID_ARG;
  if (d->accumulate && e->epilogue != MGB_EPI_F32) return MGB_ERR_INVALID_ARG;
  GemmArgs g = mk_gemm(d->dtype, d->m, d->n, d->k, d->a_major, a, d->lda, d->b_major, b, d->ldb,
                       e->epilogue, c, d->ldc);
  g.bias = bias;
  g.alpha = d->alpha;
  g.accumulate = d->accumulate;
  g.C2 = c2; g.ldc2 = e->ldc2;
  g.resid = resid; g.ldr = e->ldr;
  g.aux = aux; g.ldaux = e->ldaux;
  g.glu_block = e->glu_block;
  MGB_TRY(gemm_check(g));
  const size_t need = gemm_tf32_scratch_bytes(d->m, d->n, d->k);
  if (need > 0 && (ws == nullptr || ws_bytes < need)) return MGB_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MGB_ERR_MISALIGNED;
  MGB_TRY(check_arch());
  g.scratch = ws;
  g.scratch_bytes = ws_bytes;
  return gemm_launch(g, as_stream(stream));
}

mgb_status mgb_philox_bytes(uint64_t seed, uint64_t offset, uint64_t n, void* out, void* stream) {
  if (n > 0 && out == nullptr) return MGB_ERR_INVALID_ARG;
  MGB_TRY(check_arch());
  return philox_bytes_launch(seed, offset, n, out, as_stream(stream));
}

mgb_status mgb_dropout(int64_t rows, int64_t cols, int32_t dtype, float p, mgb_rng_state rng,
                       const void* x, int64_t ldx, void* y, int64_t ldy, void* stream) {
  if (rows < 0 || cols < 0 || !(p >= 0.0f && p < 1.0f) || dropout_threshold(p) == 0)
    return MGB_ERR_INVALID_ARG;
  if (dtype != MGB_BF16 && dtype != MGB_F32) return MGB_ERR_INVALID_ARG;
  if (rng.offset % 16 != 0) return MGB_ERR_INVALID_ARG;
  if (rows > 0 && cols > 0 && (!x || !y || ldx < cols || ldy < cols)) return MGB_ERR_INVALID_ARG;
  MGB_TRY(check_arch());
  return dropout_launch(rows, cols, dtype, p, rng.seed, rng.offset, x, ldx, y, ldy,
                        as_stream(stream));
}

mgb_status mgb_layernorm_fwd(int32_t rows, int32_t cols, int32_t dtype, float eps, const void* x,
                             const void* gamma, const void* beta, void* y, float* mean, float* rstd,
                             void* stream) {
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  if (dtype != MGB_BF16 && dtype != MGB_F32) return MGB_ERR_INVALID_ARG;
  if (rows < 0 || cols < 1 || !x || !y) return MGB_ERR_INVALID_ARG;
  const void* ps[] = {x, gamma, beta, y, mean, rstd};
  for (const void* q : ps)
    if (!aligned16(q)) return MGB_ERR_MISALIGNED;
  MGB_TRY(check_arch());
  return layernorm_fwd_launch(rows, cols, dtype, eps, x, gamma, beta, y, mean, rstd,
                              as_stream(stream));
}

size_t mgb_layernorm_bwd_ws_bytes(int32_t rows, int32_t cols) {
  if (rows < 0 || cols < 1) return 0;
  return sizeof(float) * 2 * (size_t)layernorm_bwd_parts(rows) * (size_t)cols;
}

mgb_status mgb_layernorm_bwd(int32_t rows, int32_t cols, int32_t dtype, const void* x,
                             const float* mean, const float* rstd, const void* gamma,
                             const void* dy, const void* dres, void* dx, void* dgamma, void* dbeta,
                             void* ws, size_t ws_bytes, void* stream) {
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  if (dtype != MGB_BF16 && dtype != MGB_F32) return MGB_ERR_INVALID_ARG;
  if (rows < 0 || cols < 1 || !x || !mean || !rstd || !dy || !dx) return MGB_ERR_INVALID_ARG;
  if (!gamma && (dgamma || dbeta)) return MGB_ERR_INVALID_ARG;
  const void* ps[] = {x, mean, rstd, gamma, dy, dres, dx, dgamma, dbeta, ws};
  for (const void* q : ps)
    if (!aligned16(q)) return MGB_ERR_MISALIGNED;
  const bool want = dgamma || dbeta;
  if (want && (ws == nullptr || ws_bytes < mgb_layernorm_bwd_ws_bytes(rows, cols)))
    return MGB_ERR_WORKSPACE_TOO_SMALL;
  MGB_TRY(check_arch());
  return layernorm_bwd_launch(rows, cols, dtype, x, mean, rstd, gamma, dy, dres, dx, dgamma, dbeta,
                              want ? static_cast<float*>(ws) : nullptr, layernorm_bwd_parts(rows),
                              as_stream(stream));
}

mgb_status mgb_attention_fwd(int32_t batch, int32_t seq, int32_t n_q_heads, int32_t n_kv_heads,
                             int32_t head_dim, int32_t causal, int32_t dtype, const void* q,
                             const void* k, const void* v, int64_t ld_q, int64_t ld_kv, void* o,
                             float* lse, void* stream) {
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  if (batch < 0 || seq < 1 || n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads)
    return MGB_ERR_INVALID_ARG;
  if (dtype != MGB_BF16 && dtype != MGB_F32) return MGB_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse) return MGB_ERR_INVALID_ARG;
  if (dtype == MGB_BF16 && head_dim != 64 && head_dim != 128) return MGB_ERR_UNSUPPORTED;
  if (ld_q < (int64_t)n_q_heads * head_dim || ld_kv < (int64_t)n_kv_heads * head_dim)
    return MGB_ERR_INVALID_ARG;
  const int vm = dtype == MGB_BF16 ? 8 : 1;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || ld_q % vm || ld_kv % vm)
    return MGB_ERR_MISALIGNED;
  MGB_TRY(check_arch());
  AttnArgs a{};
  a.B = batch; a.S = seq; a.nq = n_q_heads; a.nkv = n_kv_heads; a.d = head_dim;
  a.causal = causal ? 1 : 0; a.dtype = dtype;
  a.q = q; a.k = k; a.v = v; a.ld_q = ld_q; a.ld_kv = ld_kv;
  a.o = o; a.ld_o = (int64_t)n_q_heads * head_dim; a.lse = lse;
  return attention_fwd_launch(a, as_stream(stream));
}

// `table` is the shard's rows (or their gradient); `per_token` the [tokens,
// hidden] side, which (like ids) may be NULL when tokens == 0.
static mgb_status check_embedding(int32_t tokens, int32_t hidden, int32_t v0, int32_t v1,
                                  int32_t dtype, const void* ids, const void* table,
                                  const void* per_token) {
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  if (tokens < 0 || hidden < 1 || v0 < 0 || v1 <= v0) return MGB_ERR_INVALID_ARG;
  if (dtype != MGB_BF16 && dtype != MGB_F32) return MGB_ERR_INVALID_ARG;
  if (!table || (tokens > 0 && (!ids || !per_token))) return MGB_ERR_INVALID_ARG;
  if (hidden % (dtype == MGB_BF16 ? 8 : 4)) return MGB_ERR_MISALIGNED;
  if (!aligned16(table) || !aligned16(per_token) || (reinterpret_cast<uintptr_t>(ids) & 3u))
    return MGB_ERR_MISALIGNED;
  return MGB_OK;
}

mgb_status mgb_embedding_fwd(int32_t tokens, int32_t hidden, int32_t v0, int32_t v1, int32_t dtype,
                             const int32_t* ids, const void* emb_shard, void* out, void* stream) {
  MGB_TRY(check_embedding(tokens, hidden, v0, v1, dtype, ids, emb_shard, out));
  MGB_TRY(check_arch());
  return embedding_fwd_launch(tokens, hidden, dtype, v0, v1, ids, emb_shard, out,
                              as_stream(stream));
}

size_t mgb_embedding_bwd_ws_bytes(int32_t tokens, int32_t v0, int32_t v1) {
  if (tokens < 0 || v0 < 0 || v1 <= v0) return 0;
  return embedding_bwd_ws(tokens, v0, v1);
}

mgb_status mgb_embedding_bwd(int32_t tokens, int32_t hidden, int32_t v0, int32_t v1, int32_t dtype,
                             const int32_t* ids, const void* d_out, void* d_emb_shard,
                             int32_t accumulate, void* ws, size_t ws_bytes, void* stream) {
  MGB_TRY(check_embedding(tokens, hidden, v0, v1, dtype, ids, d_emb_shard, d_out));
  if (ws == nullptr) return MGB_ERR_INVALID_ARG;
  if (!aligned16(ws)) return MGB_ERR_MISALIGNED;
  if (ws_bytes < embedding_bwd_ws(tokens, v0, v1)) return MGB_ERR_WORKSPACE_TOO_SMALL;
  MGB_TRY(check_arch());
  return embedding_bwd_launch(tokens, hidden, dtype, v0, v1, ids, d_out, d_emb_shard,
                              accumulate ? 1 : 0, ws, as_stream(stream));
}

mgb_status mgb_embedding_bwd_prepare(int32_t tokens, int32_t v0, int32_t v1, const int32_t* ids,
                                     void* ws, size_t ws_bytes, mgb_embedding_bwd_plan* plan,
                                     void* stream) {
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  if (tokens < 0 || v0 < 0 || v1 <= v0 || !plan || !ws || (tokens > 0 && !ids))
    return MGB_ERR_INVALID_ARG;
  if (!aligned16(ws) || (reinterpret_cast<uintptr_t>(ids) & 3u)) return MGB_ERR_MISALIGNED;
  if (ws_bytes < embedding_bwd_ws(tokens, v0, v1)) return MGB_ERR_WORKSPACE_TOO_SMALL;
  MGB_TRY(check_arch());
  MGB_TRY(embedding_bwd_prepare_launch(tokens, v0, v1, ids, ws, as_stream(stream)));
  plan->tokens = tokens;
  plan->v0 = v0;
  plan->v1 = v1;
  plan->ws = ws;
  plan->ws_bytes = ws_bytes;
  return MGB_OK;
}

mgb_status mgb_embedding_bwd_apply(const mgb_embedding_bwd_plan* plan, int32_t hidden,
                                   int32_t dtype, const void* d_out, void* d_emb_shard,
                                   int32_t accumulate, void* stream) {
  if (!plan) return MGB_ERR_INVALID_ARG;
  // the plan's ids only decided the workspace's contents; d_out stands in for them
  MGB_TRY(check_embedding(plan->tokens, hidden, plan->v0, plan->v1, dtype, d_out, d_emb_shard,
                          d_out));
  if (!plan->ws) return MGB_ERR_INVALID_ARG;
  if (!aligned16(plan->ws)) return MGB_ERR_MISALIGNED;
  if (plan->ws_bytes < embedding_bwd_ws(plan->tokens, plan->v0, plan->v1))
    return MGB_ERR_WORKSPACE_TOO_SMALL;
  MGB_TRY(check_arch());
  return embedding_bwd_apply_launch(plan->tokens, hidden, dtype, plan->v0, plan->v1, d_out,
                                    d_emb_shard, accumulate ? 1 : 0, plan->ws, as_stream(stream));
}

size_t mgb_attention_bwd_ws_bytes(int32_t batch, int32_t seq, int32_t n_q_heads) {
  if (batch < 0 || seq < 0 || n_q_heads < 0) return 0;
  return attn_bwd_ws_bytes(batch, seq, n_q_heads);
}

mgb_status mgb_attention_bwd(int32_t batch, int32_t seq, int32_t n_q_heads, int32_t n_kv_heads,
                             int32_t head_dim, int32_t causal, int32_t dtype, const void* q,
                             const void* k, const void* v, int64_t ld_q, int64_t ld_kv,
                             const void* o, const float* lse, const void* dout, int64_t ld_do,
                             void* dq, void* dk, void* dv, int64_t ld_dq, int64_t ld_dkv, void* ws,
                             size_t ws_bytes, void* stream) {
  if (fault_injected()) return MGB_ERR_INVALID_ARG;
  if (batch < 0 || seq < 1 || n_q_heads < 1 || n_kv_heads < 1 || n_q_heads % n_kv_heads)
    return MGB_ERR_INVALID_ARG;
  if (dtype != MGB_BF16 && dtype != MGB_F32) return MGB_ERR_INVALID_ARG;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !ws) return MGB_ERR_INVALID_ARG;
  if (dtype == MGB_BF16 && head_dim != 64 && head_dim != 128) return MGB_ERR_UNSUPPORTED;
  if (dtype == MGB_F32 && (head_dim > 256 || seq > 2048)) return MGB_ERR_UNSUPPORTED;
  const int64_t wq = (int64_t)n_q_heads * head_dim, wkv = (int64_t)n_kv_heads * head_dim;
  if (ld_q < wq || ld_do < wq || ld_dq < wq || ld_kv < wkv || ld_dkv < wkv)
    return MGB_ERR_INVALID_ARG;
  const int vm = dtype == MGB_BF16 ? 8 : 1;
  const void* ps[] = {q, k, v, o, dout, dq, dk, dv, ws};
  for (const void* pp : ps)
    if (!aligned16(pp)) return MGB_ERR_MISALIGNED;
  if (ld_q % vm || ld_kv % vm || ld_do % vm || ld_dq % vm || ld_dkv % vm) return MGB_ERR_MISALIGNED;
  if (ws_bytes < attn_bwd_ws_bytes(batch, seq, n_q_heads)) return MGB_ERR_WORKSPACE_TOO_SMALL;
  MGB_TRY(check_arch());
  AttnArgs a{};
  a.B = batch; a.S = seq; a.nq = n_q_heads; a.nkv = n_kv_heads; a.d = head_dim;
  a.causal = causal ? 1 : 0; a.dtype = dtype;
  a.q = q; a.k = k; a.v = v; a.ld_q = ld_q; a.ld_kv = ld_kv;
  a.o = const_cast<void*>(o); a.ld_o = wq; a.lse = const_cast<float*>(lse);
  a.dout = dout; a.ld_do = ld_do;
  a.dq = dq; a.dk = dk; a.dv = dv; a.ld_dq = ld_dq; a.ld_dkv = ld_dkv;
  a.delta = static_cast<float*>(ws);
  return attention_bwd_launch(a, as_stream(stream));
}

}  // extern "C"
