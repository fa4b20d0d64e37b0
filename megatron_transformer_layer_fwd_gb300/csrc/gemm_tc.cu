// bf16 GEMM on the 5th-generation tensor cores (tcgen05, sm_103a).
//
// acc[m][n] = alpha * sum_k A(m,k) * B(n,k), float32 accumulation in TMEM.
// The dense contractions of the layer - QKV, output projection, fc1, fc2 and
// the vocab logits ("LLM Lab 06: build a Megatron-style Transformer Block
// from scratch", section 2; "02 - How a whole Transformer block is split",
// sections 1, 2 and 4) - and their input/weight gradients are all this product
// with one of three operand layouts:
//   forward      Y = X W^T       A K-major [M,K], B K-major [N,K]
//   input grad   dX = dY W       A K-major,       B MN-major (W stored [K_red, N])
//   weight grad  dW = dY^T X     A MN-major,      B MN-major (token dim reduced)
//
// Output tiles are BM x BN (BM = 128 rows = 128 TMEM lanes, BN columns of
// float32 accumulator). One persistent CTA per SM walks its tiles with six
// warps:
//   warp 0 lane 0  TMA producer: K-blocks of 64 into a STAGES-deep smem ring
//   warp 1 lane 0  MMA issuer: 4 x tcgen05.mma (K = 16 each) per K-block, then
//                  tcgen05.commit to the stage's "empty" barrier; tile i
//                  accumulates into TMEM buffer i & 1
//   warps 2-5      epilogue: tcgen05.ld rows out of TMEM (warp w reads lanes
//                  32*(w%4).. = tile rows), fused bias / activation / residual
//                  / activation-gradient, 16-byte global stores - while the
//                  MMAs of the next tile run into the other TMEM buffer.
// Tiles are visited in groups of row tiles sized so the group's A panel stays
// in L2 while B streams past (concurrently resident CTAs share both).
//
// Shared-memory operand layouts (128-byte swizzle, as TMA writes them):
//   K-major tile: rows of 64 bf16 (128 B); 8-row atoms of 1024 B (SBO = 1024);
//                 the k-th K=16 slice starts 32*k bytes into the tile.
//   MN-major tile: boxes of 64 MN-elements x 64 K-rows (8 KB) side by side along
//                 MN (LBO = 8192); 8-K-row atoms 1024 B apart (SBO = 1024); the
//                 k-th K=16 slice starts 2048*k bytes in.
// Every device wait is bounded (common.cuh); a wait that runs out records an
// error and the CTA drains and frees its TMEM instead of spinning forever.
#include <cudaTypedefs.h>

#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace mgb {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;

struct EpiParams {
  int M, N, K;
  int epi;
  float alpha;
  void* C;
  int64_t ldc;
  const bf16* bias;
  const bf16* resid;
  int64_t ldr;
  void* C2;
  int64_t ldc2;
  const bf16* aux;
  int64_t ldaux;
  int glu_block;
  int accumulate;
  int tiles_m, tiles_n, group_m;
  int* err;
  const int32_t* tgt;
  int tgt_v0;
  float* tgt_out;
  const float* ce_lse;
  float ce_scale;
  bf16* keep;
  int64_t ld_keep;
  uint32_t drop_thr;
  float drop_scale;
  uint64_t drop_seed, drop_offset;
  float* cpart;
  // split-K (EPI_F32 only): the K blocks are cut into k_splits ranges of
  // kb_per_split blocks; split s stores its partial product at C + s * split_stride
  int k_splits, kb_per_split;
  int64_t split_stride;
  // EPI_F32 through TMA (0 off): 1 stores, 2 reduce-adds each staged 32 x 32
  // float32 box into C (tensor map tmC)
  int c_tma;
  // bf16 outputs through TMA (0 off, 1 on): every 32-column chunk of the
  // warp's 32 rows is staged in shared memory and stored by a bulk tensor
  // copy: C (or the kept logits of EPI_CE_STATS) through tmC, C2 through tmC2
  int o_tma;
  // column chunks (EPI_CE_STATS / EPI_CE_GRAD; 0 = off): the N columns are cut
  // into chunks of n_chunk, tpc column tiles each, so no tile straddles two
  // chunks; a chunk's statistics groups start at its first column (gpc groups
  // of 128 per chunk)
  int n_chunk, tpc, gpc;
};

// Shared memory the TMA float32 epilogue stages through: two 4 KB boxes per
// epilogue warp, 1024-byte aligned after the barrier area.
constexpr int kEpiStageBytes = 4 * 2 * 4096;

template <int BN, int STAGES>
struct Cfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int TILE_BYTES = STAGE_BYTES * STAGES;
  // operand stages, 1 KB of barriers, the epilogue's TMA boxes, alignment slack
  static constexpr int SMEM_BYTES = TILE_BYTES + 1024 + kEpiStageBytes + 1024;
};

__device__ __forceinline__ void load8(const bf16* p, float (&f)[8]) {
  uint4 v = *reinterpret_cast<const uint4*>(p);
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = unpack_bf16x2(w[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void store8(bf16* p, const float* f) {
  uint4 v;
  v.x = pack_bf16x2(f[0], f[1]);
  v.y = pack_bf16x2(f[2], f[3]);
  v.z = pack_bf16x2(f[4], f[5]);
  v.w = pack_bf16x2(f[6], f[7]);
  *reinterpret_cast<uint4*>(p) = v;
}

// Bias for 32 columns starting at n (all lanes read the same addresses).
__device__ __forceinline__ void add_bias32(const bf16* bias, int n, int N, float* acc) {
  if (bias == nullptr) return;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    if (n + 8 * q < N) {
      float b[8];
      load8(bias + n + 8 * q, b);
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[8 * q + j] += b[j];
    }
  }
}

__device__ __forceinline__ void tmem_chunk(uint32_t taddr, float alpha, bool have_acc,
                                           float (&acc)[32]) {
  uint32_t r[32];
  tmem_ld32(taddr, r);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j] = have_acc ? alpha * __uint_as_float(r[j]) : 0.0f;
}

// Column sums over the warp's 32 rows (one row per lane) of 32 columns held
// as v[0..31] in each lane: a butterfly that halves the columns a lane keeps
// at each of five shuffle steps, so lane l ends with column l's sum; it is
// stored as row `row / 32` of the partials, which exist for the blocks of 32
// rows that start below M (a warp wholly past M stores nothing). Every lane of
// the warp must call it.
__device__ __forceinline__ void colsum32_store(float* part, int64_t ld, int row, int M, int c0,
                                               int ncols, float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int j = 0; j < off; ++j) {
      const float send = up ? v[j] : v[j + off];
      const float keep = up ? v[j + off] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  if ((row & ~31) < M && c0 + lane < ncols) part[(int64_t)(row >> 5) * ld + c0 + lane] = v[0];
}

// Epilogue for one thread = one output row `row` of the tile. The epilogue
// functions are kept out of line: a kernel whose epilogue code is inlined in
// full (every kind, both store paths) ran its products about 1 % slower.
template <int BN>
__device__ __noinline__ void epilogue_row(const EpiParams& p, uint32_t tmem_row, int row, int n0,
                             bool have_acc, int64_t c_off = 0, int cbase = 0, int nend = INT_MAX,
                             int pbase = 0) {
  const bool row_ok = row < p.M;
  if (p.epi == EPI_BIAS_SWIGLU) {
    const int gb = p.glu_block;
    for (int lc = 0; lc < BN; lc += 32) {
      if ((lc / gb) & 1) continue;  // visit gate chunks; the up chunk is gb further
      float g[32], u[32];
      tmem_chunk(tmem_row + lc, p.alpha, have_acc, g);
      tmem_chunk(tmem_row + lc + gb, p.alpha, have_acc, u);
      const int ng = n0 + lc, nu = ng + gb;
      if (!row_ok || ng >= p.N) continue;
      add_bias32(p.bias, ng, p.N, g);
      add_bias32(p.bias, nu, p.N, u);
      bf16* c = reinterpret_cast<bf16*>(p.C) + (int64_t)row * p.ldc;
      bf16* c2 = reinterpret_cast<bf16*>(p.C2) + (int64_t)row * p.ldc2;
      const int na = (ng / (2 * gb)) * gb + (ng % gb);
      float a[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) a[j] = g[j] * sigmoidf_(g[j]) * u[j];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        store8(c + ng + 8 * q, g + 8 * q);
        store8(c + nu + 8 * q, u + 8 * q);
        store8(c2 + na + 8 * q, a + 8 * q);
      }
    }
    return;
  }
  if (p.epi == EPI_CE_STATS) {
    // per 128-column group: running (max, sum exp) of the float32 logits in
    // the log2 domain (the sum rescaled when the max grows); no logits stored
    // (with column chunks: this tile's chunk ends at nend, its groups are
    // numbered from pbase at column cbase)
    const int NE = min(p.N, nend);
    int tcol = -1;
    if (p.tgt != nullptr && row_ok) tcol = p.tgt[row] - p.tgt_v0 - n0;
    float* pm = reinterpret_cast<float*>(p.C);
    float* ps = reinterpret_cast<float*>(p.C2);
    for (int h = 0; h < BN; h += 128) {
      float mx = -INFINITY, sum = 0.0f;
      for (int lc = h; lc < h + 128; lc += 32) {
        float acc[32];
        tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
        const int n = n0 + lc;
        if (!row_ok || n >= NE) continue;
        const int tc = tcol - lc;
        if (tc >= 0 && tc < 32 && n + tc < NE) {
          float v = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) v = (j == tc) ? acc[j] : v;
          p.tgt_out[row] = v;
        }
        if (p.keep != nullptr) {
          bf16* kp = p.keep + (int64_t)row * p.ld_keep + n;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (n + 8 * q < NE) store8(kp + 8 * q, acc + 8 * q);
        }
        float cm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          acc[j] = n + j < NE ? acc[j] * 1.4426950408889634f : -INFINITY;
          cm = fmaxf(cm, acc[j]);
        }
        if (cm > mx) {
          sum = mx == -INFINITY ? 0.0f : sum * ex2_ftz(mx - cm);
          mx = cm;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) sum += ex2_ftz(acc[j] - mx);
      }
      const int n = n0 + h;
      if (row_ok && n < NE) {
        const int64_t o = (int64_t)(pbase + (n - cbase) / 128) * p.M + row;
        pm[o] = mx * 0.6931471805599453f;
        ps[o] = sum;
      }
    }
    return;
  }
  if (p.epi == EPI_CE_GRAD) {
    // G = (softmax - onehot(target)) * scale from the float32 logits
    const int NE = min(p.N, nend);
    int tcol = -1;
    float l2 = 0.0f;
    if (row_ok) {
      tcol = p.tgt[row] - p.tgt_v0 - n0;
      l2 = p.ce_lse[row] * 1.4426950408889634f;
    }
    for (int lc = 0; lc < BN; lc += 32) {
      float acc[32];
      tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
      const int n = n0 + lc;
      if (!row_ok || n >= NE) continue;
      const int tc = tcol - lc;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float g = ex2_ftz(fmaf(acc[j], 1.4426950408889634f, -l2));
        if (j == tc) g -= 1.0f;
        acc[j] = g * p.ce_scale;
      }
      bf16* c = reinterpret_cast<bf16*>(p.C) + (int64_t)row * p.ldc + n;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (n + 8 * q < NE) store8(c + 8 * q, acc + 8 * q);
    }
    return;
  }
  if (p.epi == EPI_DGELU || p.epi == EPI_DSWIGLU) {
    // activation backward: da (the accumulator) times act'(u); rows past M
    // take no loads or stores but join the warp's bias-gradient column sums
    const int gb = p.glu_block;
    for (int lc = 0; lc < BN; lc += 32) {
      float acc[32];
      tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
      const int n = n0 + lc;
      if (n >= p.N) continue;  // the same for the whole warp
      if (p.epi == EPI_DGELU) {
        if (row_ok) {
          const bf16* ua = p.aux + (int64_t)row * p.ldaux + n;
          bf16* c = reinterpret_cast<bf16*>(p.C) + (int64_t)row * p.ldc + n;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (n + 8 * q < p.N) {
              float u[8];
              load8(ua + 8 * q, u);
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[8 * q + j] *= gelu_erf_grad(u[j]);
              store8(c + 8 * q, acc + 8 * q);
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) acc[8 * q + j] = 0.0f;
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
        }
        if (p.cpart) colsum32_store(p.cpart, p.N, row, p.M, n, p.N, acc);
      } else {
        const int i = n / gb, cc = n % gb;
        const int colg = 2 * i * gb + cc, colu = colg + gb;
        float dg[32], du[32];
        if (row_ok) {
          const bf16* ar = p.aux + (int64_t)row * p.ldaux;
          bf16* c = reinterpret_cast<bf16*>(p.C) + (int64_t)row * p.ldc;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float g[8], u[8];
            load8(ar + colg + 8 * q, g);
            load8(ar + colu + 8 * q, u);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float sg = sigmoidf_(g[j]);
              const float da = acc[8 * q + j];
              du[8 * q + j] = da * g[j] * sg;
              dg[8 * q + j] = da * u[j] * sg * (1.0f + g[j] * (1.0f - sg));
            }
            store8(c + colg + 8 * q, dg + 8 * q);
            store8(c + colu + 8 * q, du + 8 * q);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) dg[j] = du[j] = 0.0f;
        }
        if (p.cpart) {
          colsum32_store(p.cpart, 2 * (int64_t)p.N, row, p.M, colg, 2 * p.N, dg);
          colsum32_store(p.cpart, 2 * (int64_t)p.N, row, p.M, colu, 2 * p.N, du);
        }
      }
    }
    return;
  }
  // target column of this row relative to the tile (CE logits: fp32 capture)
  int tcol = -1;
  if (p.tgt != nullptr && row_ok) tcol = p.tgt[row] - p.tgt_v0 - n0;
  // every element this row stores lies in the M x N output
  if (!dcheck(row >= 0 && n0 >= 0 && (n0 & 7) == 0, p.err)) return;
  for (int lc = 0; lc < BN; lc += 32) {
    float acc[32];
    tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
    const int n = n0 + lc;
    if (!row_ok || n >= p.N) continue;
    switch (p.epi) {
      case EPI_STORE: {
        add_bias32(p.bias, n, p.N, acc);
        const int tc = tcol - lc;
        if (tc >= 0 && tc < 32 && n + tc < p.N) {
          float v = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) v = (j == tc) ? acc[j] : v;
          p.tgt_out[row] = v;
        }
        bf16* c = reinterpret_cast<bf16*>(p.C) + (int64_t)row * p.ldc + n;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (n + 8 * q < p.N) store8(c + 8 * q, acc + 8 * q);
        break;
      }
      case EPI_BIAS_GELU: {
        add_bias32(p.bias, n, p.N, acc);
        bf16* c = reinterpret_cast<bf16*>(p.C) + (int64_t)row * p.ldc + n;
        bf16* c2 = reinterpret_cast<bf16*>(p.C2) + (int64_t)row * p.ldc2 + n;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (n + 8 * q < p.N) {
            float a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) a[j] = gelu_erf(acc[8 * q + j]);
            store8(c + 8 * q, acc + 8 * q);
            store8(c2 + 8 * q, a);
          }
        }
        break;
      }
      case EPI_BIAS_RESID: {
        add_bias32(p.bias, n, p.N, acc);
        if (p.drop_thr < 256) {
          // dropout on the branch before the residual add: elements
          // row * N + n .. + 31 are stream bytes of two Philox blocks
          const uint64_t q = (p.drop_offset + (uint64_t)row * p.N + n) >> 4;
          const uint4 w0 = philox_block(p.drop_seed, q), w1 = philox_block(p.drop_seed, q + 1);
          const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
          for (int j = 0; j < 32; ++j)
            acc[j] = keep_byte(ws[j >> 2], j & 3, p.drop_thr) ? acc[j] * p.drop_scale : 0.0f;
        }
        const bf16* r = p.resid + (int64_t)row * p.ldr + n;
        bf16* c = reinterpret_cast<bf16*>(p.C) + (int64_t)row * p.ldc + n;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (n + 8 * q < p.N) {
            float x[8];
            load8(r + 8 * q, x);
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] += acc[8 * q + j];
            store8(c + 8 * q, x);
          }
        }
        break;
      }
      case EPI_F32: {
        add_bias32(p.bias, n, p.N, acc);
        float* c = reinterpret_cast<float*>(p.C) + c_off + (int64_t)row * p.ldc + n;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (n + 4 * q < p.N) {
            float4 v = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
            if (p.accumulate) {
              const float4 o = *reinterpret_cast<const float4*>(c + 4 * q);
              v.x += o.x; v.y += o.y; v.z += o.z; v.w += o.w;
            }
            *reinterpret_cast<float4*>(c + 4 * q) = v;
            acc[4 * q] = v.x; acc[4 * q + 1] = v.y; acc[4 * q + 2] = v.z; acc[4 * q + 3] = v.w;
          }
        }
        if (p.C2 != nullptr) {
          bf16* c2 = reinterpret_cast<bf16*>(p.C2) + (int64_t)row * p.ldc2 + n;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (n + 8 * q < p.N) store8(c2 + 8 * q, acc + 8 * q);
        }
        break;
      }
      default:
        break;
    }
  }
}

// EPI_F32 through TMA for one warp (rows row0 .. row0 + 31, one per lane):
// each 32-column chunk of the float32 accumulator is written to a shared
// memory box in the 128-byte swizzled layout the tensor map describes (16-byte
// chunk j of row r at r * 128 + ((j ^ (r % 8)) * 16): conflict-free vector
// stores) and one lane stores or reduce-adds the box to C with a bulk tensor
// copy; rows and columns past C's edges are clipped by the copy. Two boxes
// per warp alternate; `cnt` counts the warp's boxes so far.
template <int BN>
__device__ __noinline__ void epilogue_f32_tma(const EpiParams& p, const CUtensorMap* tmC, uint32_t tmem_row,
                                 int row0, int n0, bool have_acc, uint32_t stage, uint32_t& cnt) {
  const int lane = threadIdx.x & 31;
  for (int lc = 0; lc < BN; lc += 32) {
    float acc[32];
    tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
    const int n = n0 + lc;
    if (row0 >= p.M || n >= p.N) continue;  // the same for the whole warp
    add_bias32(p.bias, n, p.N, acc);
    const uint32_t box = stage + (cnt & 1) * 4096;
    if (lane == 0) bulk_wait_read<1>();  // the copy that last read this box is done
    __syncwarp();
    const uint32_t rb = box + lane * 128;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      st_shared_v4(rb + ((j ^ (lane & 7)) << 4), acc[4 * j], acc[4 * j + 1], acc[4 * j + 2],
                   acc[4 * j + 3]);
    fence_proxy_async();
    __syncwarp();
    if (lane == 0 && dcheck((n & 3) == 0 && row0 >= 0, p.err)) {
      if (p.c_tma == 2)
        tma_reduce_add_2d(tmC, box, n, row0);
      else
        tma_store_2d(tmC, box, n, row0);
      bulk_commit();
    }
    ++cnt;
  }
}

// One 32-column bf16 chunk of a warp's 32 rows (row row0 + lane holds v[0..31])
// through TMA: the lane's values go to a shared-memory box in the 64-byte
// swizzled layout of the tensor map (16-byte chunk j of row r at
// r * 64 + ((j ^ ((r / 2) % 4)) * 16): conflict-free vector stores), then one
// lane stores the box at column n with a bulk tensor copy, which clips rows
// and columns past the tensor's edges. Four 2 KB boxes per warp take turns;
// `cnt` counts the warp's boxes so far. Every lane of the warp calls it.
__device__ __forceinline__ void put32_tma(const CUtensorMap* tm, uint32_t stage, uint32_t& cnt,
                                          int n, int row0, const float* v, int* err) {
  const int lane = threadIdx.x & 31;
  const uint32_t box = stage + (cnt & 3) * 2048;
  if (lane == 0) bulk_wait_read<3>();  // the copy that last read this box is done
  __syncwarp();
  const uint32_t rb = box + lane * 64;
  const uint32_t sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    st_shared_v4u(rb + ((j ^ sw) << 4), pack_bf16x2(v[8 * j], v[8 * j + 1]),
                  pack_bf16x2(v[8 * j + 2], v[8 * j + 3]), pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                  pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
  fence_proxy_async();
  __syncwarp();
  if (lane == 0 && dcheck((n & 31) == 0 && n >= 0 && row0 >= 0, err)) {
    tma_store_2d(tm, box, n, row0);
    bulk_commit();
  }
  ++cnt;
}

// The bf16-output epilogues with every store through put32_tma, for one warp
// (rows row0 .. row0 + 31, lane = row): the arithmetic of epilogue_row, with
// the loads of rows past M skipped (their staged values are clipped by the
// copy). cbase / nend / pbase: the column chunk of an EPI_CE_STATS tile.
template <int BN>
__device__ __noinline__ void epilogue_tma16(const EpiParams& p, const CUtensorMap* tmC, const CUtensorMap* tmC2,
                               uint32_t tmem_row, int row0, int n0, bool have_acc, uint32_t stage,
                               uint32_t& cnt, int cbase, int nend, int pbase) {
  const int lane = threadIdx.x & 31;
  const int row = row0 + lane;
  const bool row_ok = row < p.M;
  const bool warp_in = row0 < p.M;  // the same for the whole warp
  if (p.epi == EPI_BIAS_SWIGLU) {
    const int gb = p.glu_block;
    for (int lc = 0; lc < BN; lc += 32) {
      if ((lc / gb) & 1) continue;  // visit gate chunks; the up chunk is gb further
      float g[32], u[32];
      tmem_chunk(tmem_row + lc, p.alpha, have_acc, g);
      tmem_chunk(tmem_row + lc + gb, p.alpha, have_acc, u);
      const int ng = n0 + lc, nu = ng + gb;
      if (!warp_in || ng >= p.N) continue;
      add_bias32(p.bias, ng, p.N, g);
      add_bias32(p.bias, nu, p.N, u);
      const int na = (ng / (2 * gb)) * gb + (ng % gb);
      float a[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) a[j] = g[j] * sigmoidf_(g[j]) * u[j];
      put32_tma(tmC, stage, cnt, ng, row0, g, p.err);
      put32_tma(tmC, stage, cnt, nu, row0, u, p.err);
      put32_tma(tmC2, stage, cnt, na, row0, a, p.err);
    }
    return;
  }
  if (p.epi == EPI_CE_STATS) {
    // as epilogue_row: (max, sum exp) per 128-column group from the float32
    // accumulator; the kept bf16 logits (if any) go out through TMA
    const int NE = min(p.N, nend);
    int tcol = -1;
    if (p.tgt != nullptr && row_ok) tcol = p.tgt[row] - p.tgt_v0 - n0;
    float* pm = reinterpret_cast<float*>(p.C);
    float* ps = reinterpret_cast<float*>(p.C2);
    for (int h = 0; h < BN; h += 128) {
      float mx = -INFINITY, sum = 0.0f;
      for (int lc = h; lc < h + 128; lc += 32) {
        float acc[32];
        tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
        const int n = n0 + lc;
        if (!warp_in || n >= NE) continue;
        const int tc = tcol - lc;
        if (tc >= 0 && tc < 32 && n + tc < NE) {
          float v = 0.0f;
#pragma unroll
          for (int j = 0; j < 32; ++j) v = (j == tc) ? acc[j] : v;
          p.tgt_out[row] = v;
        }
        if (p.keep != nullptr) put32_tma(tmC, stage, cnt, n, row0, acc, p.err);
        float cm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          acc[j] = n + j < NE ? acc[j] * 1.4426950408889634f : -INFINITY;
          cm = fmaxf(cm, acc[j]);
        }
        if (cm > mx) {
          sum = mx == -INFINITY ? 0.0f : sum * ex2_ftz(mx - cm);
          mx = cm;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) sum += ex2_ftz(acc[j] - mx);
      }
      const int n = n0 + h;
      if (row_ok && n < NE) {
        const int64_t o = (int64_t)(pbase + (n - cbase) / 128) * p.M + row;
        pm[o] = mx * 0.6931471805599453f;
        ps[o] = sum;
      }
    }
    return;
  }
  if (p.epi == EPI_DGELU) {
    for (int lc = 0; lc < BN; lc += 32) {
      float acc[32];
      tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
      const int n = n0 + lc;
      if (n >= p.N) continue;  // the same for the whole warp
      if (row_ok) {
        const bf16* ua = p.aux + (int64_t)row * p.ldaux + n;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (n + 8 * q < p.N) {
            float u[8];
            load8(ua + 8 * q, u);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[8 * q + j] *= gelu_erf_grad(u[j]);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[8 * q + j] = 0.0f;
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
      }
      if (warp_in) put32_tma(tmC, stage, cnt, n, row0, acc, p.err);
      if (p.cpart) colsum32_store(p.cpart, p.N, row, p.M, n, p.N, acc);
    }
    return;
  }
  if (p.epi == EPI_DSWIGLU) {
    const int gb = p.glu_block;
    for (int lc = 0; lc < BN; lc += 32) {
      float acc[32];
      tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
      const int n = n0 + lc;
      if (n >= p.N) continue;  // the same for the whole warp
      const int i = n / gb, cc = n % gb;
      const int colg = 2 * i * gb + cc, colu = colg + gb;
      float dg[32], du[32];
      if (row_ok) {
        const bf16* ar = p.aux + (int64_t)row * p.ldaux;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float g[8], u[8];
          load8(ar + colg + 8 * q, g);
          load8(ar + colu + 8 * q, u);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float sg = sigmoidf_(g[j]);
            const float da = acc[8 * q + j];
            du[8 * q + j] = da * g[j] * sg;
            dg[8 * q + j] = da * u[j] * sg * (1.0f + g[j] * (1.0f - sg));
          }
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) dg[j] = du[j] = 0.0f;
      }
      if (warp_in) {
        put32_tma(tmC, stage, cnt, colg, row0, dg, p.err);
        put32_tma(tmC, stage, cnt, colu, row0, du, p.err);
      }
      if (p.cpart) {
        colsum32_store(p.cpart, 2 * (int64_t)p.N, row, p.M, colg, 2 * p.N, dg);
        colsum32_store(p.cpart, 2 * (int64_t)p.N, row, p.M, colu, 2 * p.N, du);
      }
    }
    return;
  }
  // EPI_STORE, EPI_BIAS_GELU, EPI_BIAS_RESID: one loop each, so the loop a
  // tile runs holds only its own epilogue's instructions
  if (p.epi == EPI_STORE) {
    int tcol = -1;
    if (p.tgt != nullptr && row_ok) tcol = p.tgt[row] - p.tgt_v0 - n0;
    for (int lc = 0; lc < BN; lc += 32) {
      float acc[32];
      tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
      const int n = n0 + lc;
      if (!warp_in || n >= p.N) continue;
      add_bias32(p.bias, n, p.N, acc);
      const int tc = tcol - lc;
      if (tc >= 0 && tc < 32 && n + tc < p.N) {
        float v = 0.0f;
#pragma unroll
        for (int j = 0; j < 32; ++j) v = (j == tc) ? acc[j] : v;
        p.tgt_out[row] = v;
      }
      put32_tma(tmC, stage, cnt, n, row0, acc, p.err);
    }
    return;
  }
  if (p.epi == EPI_BIAS_GELU) {
    for (int lc = 0; lc < BN; lc += 32) {
      float acc[32];
      tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
      const int n = n0 + lc;
      if (!warp_in || n >= p.N) continue;
      add_bias32(p.bias, n, p.N, acc);
      float a[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) a[j] = gelu_erf(acc[j]);
      put32_tma(tmC, stage, cnt, n, row0, acc, p.err);
      put32_tma(tmC2, stage, cnt, n, row0, a, p.err);
    }
    return;
  }
  // EPI_BIAS_RESID
  for (int lc = 0; lc < BN; lc += 32) {
    float acc[32];
    tmem_chunk(tmem_row + lc, p.alpha, have_acc, acc);
    const int n = n0 + lc;
    if (!warp_in || n >= p.N) continue;
    add_bias32(p.bias, n, p.N, acc);
    if (p.drop_thr < 256) {
      const uint64_t q = (p.drop_offset + (uint64_t)row * p.N + n) >> 4;
      const uint4 w0 = philox_block(p.drop_seed, q), w1 = philox_block(p.drop_seed, q + 1);
      const uint32_t ws[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
      for (int j = 0; j < 32; ++j)
        acc[j] = keep_byte(ws[j >> 2], j & 3, p.drop_thr) ? acc[j] * p.drop_scale : 0.0f;
    }
    if (row_ok) {
      const bf16* r = p.resid + (int64_t)row * p.ldr + n;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (n + 8 * q < p.N) {
          float x[8];
          load8(r + 8 * q, x);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[8 * q + j] += x[j];
        }
      }
    }
    put32_tma(tmC, stage, cnt, n, row0, acc, p.err);
  }
}

// Tile `tile` of the grouped raster: group_m row tiles per group, the row
// tile advancing fastest inside a group.
__device__ __forceinline__ void tile_origin(const EpiParams& p, int tile, int bn, int& m0,
                                            int& n0, int bm = BM) {
  const int per_group = p.group_m * p.tiles_n;
  const int group = tile / per_group;
  const int first_m = group * p.group_m;
  const int gm = min(p.tiles_m - first_m, p.group_m);
  const int in_group = tile - group * per_group;
  m0 = (first_m + in_group % gm) * bm;
  n0 = (in_group / gm) * bn;
}

// Tile `tile` of the split-K grid: splits outermost (a wave of CTAs works on
// one K range, so its A and B slices are shared in L2), then the grouped
// raster of output tiles. [kb0, kb1) are the tile's K blocks.
__device__ __forceinline__ void tile_decode(const EpiParams& p, int tile, int bn, int num_k,
                                            int& m0, int& n0, int& kb0, int& kb1, int& split,
                                            int bm = BM) {
  const int per_split = p.tiles_m * p.tiles_n;
  split = tile / per_split;
  tile_origin(p, tile - split * per_split, bn, m0, n0, bm);
  if (p.n_chunk > 0) {
    // column tile n0 / bn = tile j of chunk c
    const int jn = n0 / bn, c = jn / p.tpc;
    n0 = c * p.n_chunk + (jn - c * p.tpc) * bn;
  }
  kb0 = split * p.kb_per_split;
  kb1 = min(num_k, kb0 + p.kb_per_split);
}

// Columns the tile grid spans: N, or with column chunks the whole chunk grid
// (a ragged last chunk can hold a tile that starts past N: its loads read the
// fill value and its epilogue stores nothing).
__device__ __forceinline__ int n_extent(const EpiParams& p) {
  return p.n_chunk > 0 ? (p.N + p.n_chunk - 1) / p.n_chunk * p.n_chunk : p.N;
}

// Column chunk of a tile at n0 (column chunks on): first column, end, first
// statistics group.
__device__ __forceinline__ void chunk_of(const EpiParams& p, int n0, int& cbase, int& nend,
                                         int& pbase) {
  if (p.n_chunk > 0) {
    const int c = n0 / p.n_chunk;
    cbase = c * p.n_chunk;
    nend = cbase + p.n_chunk;
    pbase = c * p.gpc;
  } else {
    cbase = 0;
    nend = INT_MAX;
    pbase = 0;
  }
}

// Persistent and warp-specialised: one CTA per SM walks the tiles
// blockIdx.x, blockIdx.x + gridDim.x, ... Six warps:
//   warp 0 (one lane)  TMA producer over every k-block of every tile of the CTA
//   warp 1 (one lane)  MMA issuer: tile i accumulates into TMEM buffer i & 1
//   warps 2-5          epilogue of tile i from buffer i & 1 (warp w reads TMEM
//                      lanes 32*(w%4)..) while tile i+1's MMAs fill the other
// The two accumulators take 2*BN TMEM columns. A wait that runs out sets a
// shared abort flag; every role then leaves its loop (no CTA barrier inside
// the loops) and the CTA meets once more to free TMEM.
template <int BN, int STAGES, int A_MN, int B_MN>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA,
                   const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmC2,
                   const __grid_constant__ EpiParams p) {
  using C = Cfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::TILE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t tiles = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t accf0 = empty0 + 8 * STAGES;  // accumulator ready, per buffer
  const uint32_t acce0 = accf0 + 16;           // accumulator drained, per buffer

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_k = (p.K + BK - 1) / BK;
  const int total = p.tiles_m * p.tiles_n * p.k_splits;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 4);  // one arrival per epilogue warp
    }
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 0) tmem_alloc(smem_u32(tmem_slot), 2 * BN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      uint32_t kg = 0;  // k-blocks issued by this CTA so far (ring position)
      for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x) {
        int m0, n0, kb0, kb1, sp;
        tile_decode(p, tile, BN, num_k, m0, n0, kb0, kb1, sp);
        for (int kb = kb0; kb < kb1; ++kb, ++kg) {
          const int s = kg % STAGES;
          if (!mbar_wait(empty0 + 8 * s, ((kg / STAGES) & 1) ^ 1, p.err)) {
            *abort = 1;
            break;
          }
          const uint32_t sa = tiles + s * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
          const uint32_t fb = full0 + 8 * s;
          const int k0 = kb * BK;
          // the tile lies in the problem and every TMA x coordinate is a
          // multiple of 8 bf16 (16 bytes); a failed check skips the copies
          // (the stage then never fills and the bounded waits end the kernel)
          if (!dcheck(m0 < p.M && n0 < n_extent(p) && kb < num_k && (k0 & 7) == 0 &&
                          (m0 & 7) == 0 && (n0 & 7) == 0,
                      p.err)) {
            *abort = 1;
            break;
          }
          mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
          if (A_MN == 0) {
            tma_load_2d(sa, &tmA, k0, m0, fb);
          } else {
            tma_load_2d(sa, &tmA, m0, k0, fb);
            tma_load_2d(sa + 8192, &tmA, m0 + 64, k0, fb);
          }
          if (B_MN == 0) {
            tma_load_2d(sb, &tmB, k0, n0, fb);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + 8192 * j, &tmB, n0 + 64 * j, k0, fb);
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, A_MN, B_MN);
      uint32_t kg = 0;
      int t = 0;  // tiles of this CTA so far
      for (int tile = blockIdx.x; tile < total && !*abort; tile += gridDim.x, ++t) {
        const int buf = t & 1;
        if (!mbar_wait(acce0 + 8 * buf, ((t >> 1) & 1) ^ 1, p.err)) {
          *abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + buf * BN;
        bool good = true;
        int m0, n0, kb0, kb1, sp;
        tile_decode(p, tile, BN, num_k, m0, n0, kb0, kb1, sp);
        for (int kb = kb0; kb < kb1; ++kb, ++kg) {
          const int s = kg % STAGES;
          if (!mbar_wait(full0 + 8 * s, (kg / STAGES) & 1, p.err)) {
            good = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = tiles + s * C::STAGE_BYTES;
          const uint32_t sb = sa + C::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? smem_desc_sw128(sa + 2048 * kk, 8192, 1024)
                                     : smem_desc_sw128(sa + 32 * kk, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sb + 2048 * kk, 8192, 1024)
                                     : smem_desc_sw128(sb + 32 * kk, 16, 1024);
            tc_mma_f16(acc, ad, bd, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
          }
          tc_commit(empty0 + 8 * s);
        }
        if (!good) {
          *abort = 1;
          break;
        }
        tc_commit(accf0 + 8 * buf);
      }
    }
  } else {
    // ---------------- epilogue warps 2..5
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const uint32_t stage = tiles + C::TILE_BYTES + 1024 + q * 8192;
    uint32_t cnt = 0;
    int t = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++t) {
      const int buf = t & 1;
      const bool ready = !*abort && mbar_wait(accf0 + 8 * buf, (t >> 1) & 1, p.err);
      if (!__all_sync(0xffffffffu, ready)) {  // warp-uniform exit
        *abort = 1;
        break;
      }
      tc_fence_after();
      int m0, n0, kb0, kb1, sp;
      tile_decode(p, tile, BN, num_k, m0, n0, kb0, kb1, sp);
      const uint32_t trow = tmem + buf * BN + ((uint32_t)(q * 32) << 16);
      if (p.c_tma) {
        epilogue_f32_tma<BN>(p, &tmC, trow, m0 + q * 32, n0, kb1 > kb0, stage, cnt);
      } else {
        int cb, ne, pb;
        chunk_of(p, n0, cb, ne, pb);
        if (p.o_tma)
          epilogue_tma16<BN>(p, &tmC, &tmC2, trow, m0 + q * 32, n0, kb1 > kb0, stage, cnt, cb, ne,
                             pb);
        else
          epilogue_row<BN>(p, trow, m0 + q * 32 + lane, n0, kb1 > kb0, sp * p.split_stride, cb,
                           ne, pb);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acce0 + 8 * buf);
    }
    // this warp's copies complete before exit
    if ((p.c_tma || p.o_tma) && lane == 0) bulk_wait<0>();
  }

  __syncthreads();
  if (*abort && threadIdx.x == 0) {
    // give copies and MMAs still in flight time to land (bounded)
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 10000000ull) {
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * BN);
  }
}

// CTA-pair variant (cluster of two CTAs on two SMs): 256 x 256 output tiles,
// one per pair. Each CTA stages its 128 rows of A and its 128 columns of B
// (32 KB per 64-wide K block instead of 48 KB for a 128 x 256 tile on one SM,
// so one SM's shared memory holds more K blocks in flight and each SM pulls a
// third fewer bytes through L2). The leader (rank 0) issues M = 256, N = 256
// tcgen05.mma.cta_group::2 products; each CTA's TMEM holds the float32
// accumulator of its own 128 rows, and each CTA runs the epilogue of its rows.
// Barriers, at the same offsets in both CTAs:
//   full[s]   leader only: both CTAs' TMA bytes of stage s (the leader expects
//             them all; the peer's copies signal the leader's barrier)
//   empty[s]  both: the leader's commit, multicast, frees stage s in both
//   accf[b]   both: the leader's commit, multicast: accumulator b complete
//   acce[b]   leader only: the 4 epilogue warps of both CTAs have read b
template <int STAGES, int A_MN, int B_MN>
__global__ void __launch_bounds__(192, 1)
    gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC,
                        const __grid_constant__ CUtensorMap tmC2,
                        const __grid_constant__ EpiParams p) {
  constexpr int BNP = 256, HALF = 128;
  constexpr int A_BYTES = HALF * BK * 2, B_BYTES = HALF * BK * 2;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t tiles = smem_u32(smem);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8 * STAGES;
  const uint32_t accf0 = empty0 + 8 * STAGES;
  const uint32_t acce0 = accf0 + 16;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int num_k = (p.K + BK - 1) / BK;
  const int total = p.tiles_m * p.tiles_n * p.k_splits;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, 8);  // 4 epilogue warps in each CTA
    }
    fence_mbar_init();
    *abort = 0;
  }
  if (warp == 0) tmem_alloc_pair(smem_u32(tmem_slot), 2 * BNP);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised before any remote signal
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs)
      uint32_t kg = 0;
      for (int tile = pair; tile < total && !*abort; tile += npairs) {
        int m0, n0, kb0, kb1, sp;
        tile_decode(p, tile, BNP, num_k, m0, n0, kb0, kb1, sp, 2 * HALF);
        const int ma = m0 + HALF * (int)rank, nb = n0 + HALF * (int)rank;
        for (int kb = kb0; kb < kb1; ++kb, ++kg) {
          const int s = kg % STAGES;
          if (!mbar_wait(empty0 + 8 * s, ((kg / STAGES) & 1) ^ 1, p.err)) {
            *abort = 1;
            break;
          }
          const uint32_t sa = tiles + s * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
          const uint32_t fb = mapa_shared(full0 + 8 * s, 0);
          const int k0 = kb * BK;
          if (!dcheck(m0 < p.M && n0 < n_extent(p) && kb < num_k && (k0 & 7) == 0 &&
                          (ma & 7) == 0 && (nb & 7) == 0,
                      p.err)) {
            *abort = 1;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(full0 + 8 * s, 2 * STAGE_BYTES);
          if (A_MN == 0) {
            tma_load_2d_pair(sa, &tmA, k0, ma, fb);
          } else {
            tma_load_2d_pair(sa, &tmA, ma, k0, fb);
            tma_load_2d_pair(sa + 8192, &tmA, ma + 64, k0, fb);
          }
          if (B_MN == 0) {
            tma_load_2d_pair(sb, &tmB, k0, nb, fb);
          } else {
            tma_load_2d_pair(sb, &tmB, nb, k0, fb);
            tma_load_2d_pair(sb + 8192, &tmB, nb + 64, k0, fb);
          }
        }
      }
      // drain: every stage released once more, so no multicast arrival on
      // this CTA's empty barriers is still on its way when the CTA exits
      for (int i = 0; i < STAGES && !*abort; ++i, ++kg) {
        const int s = kg % STAGES;
        if (!mbar_wait(empty0 + 8 * s, ((kg / STAGES) & 1) ^ 1, p.err)) *abort = 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (leader)
      constexpr uint32_t idesc = idesc_bf16_f32(2 * HALF, BNP, A_MN, B_MN);
      uint32_t kg = 0;
      int t = 0;
      for (int tile = pair; tile < total && !*abort; tile += npairs, ++t) {
        const int buf = t & 1;
        if (!mbar_wait(acce0 + 8 * buf, ((t >> 1) & 1) ^ 1, p.err)) {
          *abort = 1;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem + buf * BNP;
        bool good = true;
        int m0, n0, kb0, kb1, sp;
        tile_decode(p, tile, BNP, num_k, m0, n0, kb0, kb1, sp, 2 * HALF);
        for (int kb = kb0; kb < kb1; ++kb, ++kg) {
          const int s = kg % STAGES;
          if (!mbar_wait(full0 + 8 * s, (kg / STAGES) & 1, p.err)) {
            good = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = tiles + s * STAGE_BYTES;
          const uint32_t sb = sa + A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? smem_desc_sw128(sa + 2048 * kk, 8192, 1024)
                                     : smem_desc_sw128(sa + 32 * kk, 16, 1024);
            const uint64_t bd = B_MN ? smem_desc_sw128(sb + 2048 * kk, 8192, 1024)
                                     : smem_desc_sw128(sb + 32 * kk, 16, 1024);
            tc_mma_f16_pair(acc, ad, bd, idesc, (kb != kb0 || kk != 0) ? 1u : 0u);
          }
          tc_commit_pair_mc(empty0 + 8 * s, 3);
        }
        if (!good) {
          *abort = 1;
          break;
        }
        tc_commit_pair_mc(accf0 + 8 * buf, 3);
      }
    }
  } else {
    // ---------------- epilogue warps 2..5 (both CTAs: this CTA's 128 rows)
    const int q = warp & 3;
    const uint32_t stage = tiles + STAGES * STAGE_BYTES + 1024 + q * 8192;
    uint32_t cnt = 0;
    int t = 0;
    for (int tile = pair; tile < total; tile += npairs, ++t) {
      const int buf = t & 1;
      const bool ready = !*abort && mbar_wait(accf0 + 8 * buf, (t >> 1) & 1, p.err);
      if (!__all_sync(0xffffffffu, ready)) {
        *abort = 1;
        break;
      }
      tc_fence_after();
      int m0, n0, kb0, kb1, sp;
      tile_decode(p, tile, BNP, num_k, m0, n0, kb0, kb1, sp, 2 * HALF);
      const uint32_t trow = tmem + buf * BNP + ((uint32_t)(q * 32) << 16);
      const int r0 = m0 + HALF * (int)rank + q * 32;
      if (p.c_tma) {
        epilogue_f32_tma<BNP>(p, &tmC, trow, r0, n0, kb1 > kb0, stage, cnt);
      } else {
        int cb, ne, pb;
        chunk_of(p, n0, cb, ne, pb);
        if (p.o_tma)
          epilogue_tma16<BNP>(p, &tmC, &tmC2, trow, r0, n0, kb1 > kb0, stage, cnt, cb, ne, pb);
        else
          epilogue_row<BNP>(p, trow, r0 + lane, n0, kb1 > kb0, sp * p.split_stride, cb, ne, pb);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(acce0 + 8 * buf, 0));
    }
    // this warp's copies complete before exit
    if ((p.c_tma || p.o_tma) && lane == 0) bulk_wait<0>();
  }

  __syncthreads();
  if (*abort && threadIdx.x == 0) {
    const uint64_t t0 = global_ns();
    while (global_ns() - t0 < 10000000ull) {
    }
  }
  tc_fence_before();
  cluster_sync();  // neither CTA frees TMEM or exits while its peer may still signal it
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 2 * BNP);
  }
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2-D bf16 tensor map: inner dimension `inner` (contiguous), `outer` rows of
// stride ld elements; box = box_inner x box_outer, 128-byte swizzle, zero fill.
bool make_tmap(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, int64_t ld,
               uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D float32 tensor map of C for the TMA epilogue: boxes of 32 columns x 32
// rows, 128-byte swizzle.
bool make_tmap_f32(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, int64_t ld) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D bf16 tensor map of an epilogue output for put32_tma: boxes of 32
// columns x 32 rows, 64-byte swizzle.
bool make_tmap_out(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer, int64_t ld) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The epilogue's output maps: C (or the kept logits) and C2 for the TMA
// epilogues (o_tma), C as float32 boxes for the float32 TMA epilogue (c_tma);
// maps that are not read are copies of `fill`.
bool make_out_maps(const GemmArgs& g, const EpiParams& ep, const CUtensorMap& fill, CUtensorMap* tc,
                   CUtensorMap* tc2) {
  *tc = fill;
  *tc2 = fill;
  if (ep.c_tma) return make_tmap_f32(tc, g.C, g.N, g.M, g.ldc);
  if (!ep.o_tma) return true;
  switch (g.epi) {
    case EPI_CE_STATS:
      return make_tmap_out(tc, g.keep, g.N, g.M, g.ld_keep);
    case EPI_DSWIGLU:
      return make_tmap_out(tc, g.C, 2 * (uint64_t)g.N, g.M, g.ldc);
    case EPI_BIAS_SWIGLU:
      return make_tmap_out(tc, g.C, g.N, g.M, g.ldc) &&
             make_tmap_out(tc2, g.C2, g.N / 2, g.M, g.ldc2);
    case EPI_BIAS_GELU:
      return make_tmap_out(tc, g.C, g.N, g.M, g.ldc) && make_tmap_out(tc2, g.C2, g.N, g.M, g.ldc2);
    default:
      return make_tmap_out(tc, g.C, g.N, g.M, g.ldc);
  }
}

// One persistent CTA per SM (the kernel's shared memory allows one), never
// more CTAs than tiles.
int persistent_grid(const EpiParams& ep) {
  const long total = (long)ep.tiles_m * ep.tiles_n * ep.k_splits;
  return (int)std::max(1L, std::min<long>(total, device_sm_count()));
}

template <int BN, int STAGES, int A_MN, int B_MN>
mgb_status launch_variant(const GemmArgs& g, const EpiParams& ep, cudaStream_t st) {
  using C = Cfg<BN, STAGES>;
  auto kern = gemm_tc_kernel<BN, STAGES, A_MN, B_MN>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES) !=
      cudaSuccess)
    return MGB_ERR_CUDA;
  CUtensorMap ta, tb, tc;
  if (g.K == 0) {
    // no K blocks: the kernel writes the epilogue of a zero accumulator and
    // never reads the operands; encode harmless maps over the output buffer
    const bool ok0 = make_tmap(&ta, g.C, 64, 64, 64, 64, 64) && make_tmap(&tb, g.C, 64, 64, 64, 64, 64);
    if (!ok0) return MGB_ERR_CUDA;
  } else {
    bool ok = A_MN ? make_tmap(&ta, g.A, g.M, g.K, g.lda, 64, 64)
                   : make_tmap(&ta, g.A, g.K, g.M, g.lda, 64, BM);
    ok = ok && (B_MN ? make_tmap(&tb, g.B, g.N, g.K, g.ldb, 64, 64)
                     : make_tmap(&tb, g.B, g.K, g.N, g.ldb, 64, BN));
    if (!ok) return MGB_ERR_CUDA;
  }
  CUtensorMap tc2;
  if (!make_out_maps(g, ep, ta, &tc, &tc2)) return MGB_ERR_CUDA;
  LaunchScope scope(g.prof_kind >= 0 ? g.prof_kind
                               : (A_MN ? PROF_GEMM_WGRAD : (B_MN ? PROF_GEMM_DGRAD : PROF_GEMM_FWD)),
                    st);
  kern<<<persistent_grid(ep), 192, C::SMEM_BYTES, st>>>(ta, tb, tc, tc2, ep);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

constexpr int PAIR_STAGES = 6;
constexpr int pair_smem_bytes() {
  return PAIR_STAGES * 2 * (128 * BK * 2) + 1024 + kEpiStageBytes + 1024;
}

template <int A_MN, int B_MN>
mgb_status launch_pair_variant(const GemmArgs& g, const EpiParams& ep, cudaStream_t st) {
  auto kern = gemm_tc_pair_kernel<PAIR_STAGES, A_MN, B_MN>;
  constexpr int smem = pair_smem_bytes();
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return MGB_ERR_CUDA;
  CUtensorMap ta, tb, tc;
  bool ok = A_MN ? make_tmap(&ta, g.A, g.M, g.K, g.lda, 64, 64)
                 : make_tmap(&ta, g.A, g.K, g.M, g.lda, 64, 128);
  ok = ok && (B_MN ? make_tmap(&tb, g.B, g.N, g.K, g.ldb, 64, 64)
                   : make_tmap(&tb, g.B, g.K, g.N, g.ldb, 64, 128));
  CUtensorMap tc2;
  ok = ok && make_out_maps(g, ep, ta, &tc, &tc2);
  if (!ok) return MGB_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // persistent: as many pairs as can be resident at once (one CTA per SM),
  // never more than there are tiles
  static int max_pairs[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (max_pairs[dev] == 0) {
    int n = 0;
    cfg.gridDim = dim3(2 * (device_sm_count() / 2), 1, 1);
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = device_sm_count() / 2;
    }
    max_pairs[dev] = n;
  }
  const long total = (long)ep.tiles_m * ep.tiles_n * ep.k_splits;
  const int pairs = (int)std::max(1L, std::min<long>(total, max_pairs[dev]));
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  LaunchScope scope(g.prof_kind >= 0 ? g.prof_kind
                               : (A_MN ? PROF_GEMM_WGRAD : (B_MN ? PROF_GEMM_DGRAD : PROF_GEMM_FWD)),
                    st);
  if (cudaLaunchKernelEx(&cfg, kern, ta, tb, tc, tc2, ep) != cudaSuccess) return MGB_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

// Column tiles of width bn, per column chunk when chunks are on.
void set_tiles_n(EpiParams& ep, int N, int bn) {
  if (ep.n_chunk > 0) {
    ep.tpc = (ep.n_chunk + bn - 1) / bn;
    ep.gpc = (ep.n_chunk + 127) / 128;
    ep.tiles_n = (N + ep.n_chunk - 1) / ep.n_chunk * ep.tpc;
  } else {
    ep.tiles_n = (N + bn - 1) / bn;
  }
}

// Row tiles per raster group. Tiles are visited group by group, the row tile
// advancing fastest inside a group, so a group's A rows stay in L2 while its
// B columns stream past. With the K range of one split (kb_per_split blocks):
// if all of B fits comfortably in L2 (e.g. a weight gradient's short token
// panel), one row tile per group reads every A panel once and keeps B
// resident; if all of A fits, one group of all rows reads B once; otherwise
// groups of about 48 MB of A rows.
int raster_group(const EpiParams& ep, int M, int N, int bm, int min_g, int max_g) {
  const long k_eff = (long)ep.kb_per_split * BK;
  const long fits = 40L << 20;
  if ((long)N * k_eff * 2 <= fits) return 1;
  if ((long)M * k_eff * 2 <= fits) return ep.tiles_m;
  // split-K with few row tiles: each wave spans every row tile and the
  // fewest column tiles, so the concurrent tiles (which walk their K range
  // together) share the most A and B slices in L2
  if (ep.k_splits > 1 && ep.tiles_m <= 16) return ep.tiles_m;
  const long panel = (long)bm * (k_eff > 0 ? k_eff : 1) * 2;
  const int g = (int)std::max((long)min_g, std::min((long)max_g, (48L << 20) / panel));
  return std::min(g, ep.tiles_m);
}

mgb_status launch_pair(const GemmArgs& g, EpiParams ep, cudaStream_t st) {
  ep.tiles_m = (g.M + 255) / 256;
  set_tiles_n(ep, g.N, 256);
  ep.group_m = raster_group(ep, g.M, g.N, 256, 2, 32);
  if (!g.a_mn && !g.b_mn) return launch_pair_variant<0, 0>(g, ep, st);
  if (!g.a_mn && g.b_mn) return launch_pair_variant<0, 1>(g, ep, st);
  if (g.a_mn && g.b_mn) return launch_pair_variant<1, 1>(g, ep, st);
  return launch_pair_variant<1, 0>(g, ep, st);
}

template <int BN, int STAGES>
mgb_status launch_bn(const GemmArgs& g, EpiParams ep, cudaStream_t st) {
  ep.tiles_m = (g.M + BM - 1) / BM;
  set_tiles_n(ep, g.N, BN);
  ep.group_m = raster_group(ep, g.M, g.N, BM, 4, 64);
  if (!g.a_mn && !g.b_mn) return launch_variant<BN, STAGES, 0, 0>(g, ep, st);
  if (!g.a_mn && g.b_mn) return launch_variant<BN, STAGES, 0, 1>(g, ep, st);
  if (g.a_mn && g.b_mn) return launch_variant<BN, STAGES, 1, 1>(g, ep, st);
  return launch_variant<BN, STAGES, 1, 0>(g, ep, st);
}

}  // namespace

// 2-D bf16 tensor map with 128-byte swizzle and zero fill (shared with the
// attention kernels).
CUresult tmap_encode_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                             int64_t ld, uint32_t box_inner, uint32_t box_outer) {
  return make_tmap(tm, base, inner, outer, ld, box_inner, box_outer) ? CUDA_SUCCESS
                                                                     : CUDA_ERROR_INVALID_VALUE;
}

// 2-D float32 tensor map with 128-byte swizzle (box_inner 32 or fewer words).
CUresult tmap_encode_f32_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                            int64_t ld, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_INITIALIZED;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// 2-D uint32 tensor map without swizzle (box rows of box_inner words).
CUresult tmap_encode_u32_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t outer,
                            int64_t ld, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encode_fn();
  if (!fn) return CUDA_ERROR_NOT_INITIALIZED;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 4};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Whether the bf16 outputs of this product go through TMA (epilogue_tma16):
// the bf16-output epilogues with 32-column-aligned output chunks (gate/up
// blocks and vocab chunks multiples of 32), rows that are multiples of 16
// bytes apart, 16-byte-aligned outputs, no split over K. MGB_GEMM_TMA_OUT=0
// keeps every store on the per-thread path.
bool out_tma_ok(const GemmArgs& g, int n_chunk) {
  const char* e = getenv("MGB_GEMM_TMA_OUT");
  if (e != nullptr && e[0] == '0') return false;
  if (g.k_splits > 1) return false;
  auto al = [](const void* q, int64_t ld) {
    return q != nullptr && (reinterpret_cast<uintptr_t>(q) & 15u) == 0 && ld % 8 == 0;
  };
  switch (g.epi) {
    case EPI_STORE:
    case EPI_BIAS_RESID:
    case EPI_DGELU:
      return al(g.C, g.ldc);
    case EPI_DSWIGLU:
      return al(g.C, g.ldc) && g.glu_block % 32 == 0;
    case EPI_BIAS_GELU:
      return al(g.C, g.ldc) && al(g.C2, g.ldc2);
    case EPI_BIAS_SWIGLU:
      return al(g.C, g.ldc) && al(g.C2, g.ldc2) && g.glu_block % 32 == 0;
    case EPI_CE_STATS:
      return g.keep != nullptr && al(g.keep, g.ld_keep) && n_chunk % 32 == 0;
    default:
      return false;
  }
}

mgb_status gemm_tc_launch(const GemmArgs& g, cudaStream_t st) {
  EpiParams ep{};
  ep.M = g.M; ep.N = g.N; ep.K = g.K;
  ep.epi = g.epi; ep.alpha = g.alpha;
  ep.C = g.C; ep.ldc = g.ldc;
  ep.bias = reinterpret_cast<const bf16*>(g.bias);
  ep.resid = reinterpret_cast<const bf16*>(g.resid); ep.ldr = g.ldr;
  ep.C2 = g.C2; ep.ldc2 = g.ldc2;
  ep.aux = reinterpret_cast<const bf16*>(g.aux); ep.ldaux = g.ldaux;
  ep.glu_block = g.glu_block; ep.accumulate = g.accumulate;
  ep.err = device_error_word();
  ep.tgt = (g.epi == EPI_STORE || g.epi == EPI_CE_STATS || g.epi == EPI_CE_GRAD) ? g.tgt : nullptr;
  ep.ce_lse = g.ce_lse;
  ep.ce_scale = g.ce_scale;
  ep.keep = static_cast<bf16*>(g.keep);
  ep.ld_keep = g.ld_keep;
  ep.drop_thr = g.drop_thr;
  ep.drop_scale = g.drop_scale;
  ep.drop_seed = g.drop_seed;
  ep.drop_offset = g.drop_offset;
  ep.tgt_v0 = g.tgt_v0;
  ep.tgt_out = g.tgt_out;
  ep.cpart = (g.epi == EPI_DGELU || g.epi == EPI_DSWIGLU) ? g.colsum_part : nullptr;
  ep.c_tma = (g.epi == EPI_F32 && g.f32_tma) ? (g.accumulate ? 2 : 1) : 0;
  ep.n_chunk = (g.epi == EPI_CE_STATS || g.epi == EPI_CE_GRAD) && g.n_chunk < g.N ? g.n_chunk : 0;
  ep.tpc = ep.gpc = 0;
  ep.o_tma = out_tma_ok(g, ep.n_chunk) ? 1 : 0;
  const int num_k = (g.K + BK - 1) / BK;
  ep.k_splits = 1;
  ep.kb_per_split = num_k;
  ep.split_stride = 0;
  if (g.k_splits > 1 && num_k > 1) {
    ep.kb_per_split = (num_k + g.k_splits - 1) / g.k_splits;
    ep.k_splits = (num_k + ep.kb_per_split - 1) / ep.kb_per_split;  // no empty range
    ep.split_stride = g.split_stride;
  }
  // Tile: 256 x 256 on a CTA pair when there are enough such tiles to fill
  // the GPU; else 128 x 256 on one SM, or 128 x 128 when the problem is too
  // narrow to fill the GPU with 256 columns. MGB_GEMM_PAIR=0 / =1 turns the
  // pair tile off / on whenever K > 0 (tests cover both on small shapes).
  const long tiles256 = (long)((g.M + BM - 1) / BM) * ((g.N + 255) / 256);
  const long pair_tiles = (long)((g.M + 255) / 256) * ((g.N + 255) / 256);
  const char* pe = getenv("MGB_GEMM_PAIR");
  const int force = pe == nullptr ? -1 : (pe[0] == '1' ? 1 : (pe[0] == '0' ? 0 : -1));
  const bool pair = g.K > 0 && (force == 1 || (force == -1 && g.M > 128 && g.N > 128 &&
                                               pair_tiles * ep.k_splits >= device_sm_count() / 2));
  if (pair) return launch_pair(g, ep, st);
  if (g.epi == EPI_BIAS_SWIGLU || (tiles256 >= 148 && g.N > 128))
    return launch_bn<256, 4>(g, ep, st);
  return launch_bn<128, 6>(g, ep, st);
}

int gemm_splitk_count(int M, int N, int K, int max_splits) {
  const long tiles = (long)((M + 255) / 256) * ((N + 255) / 256);
  const int num_k = (K + BK - 1) / BK;
  const int npairs = std::max(1, device_sm_count() / 2);
  if (tiles <= 0 || num_k < 16) return 1;
  // fraction of the pair slots busy over the waves a split count needs
  auto fill = [&](int s) {
    const long t = tiles * s;
    const long waves = (t + npairs - 1) / npairs;
    return (double)t / (double)(waves * npairs);
  };
  int best = 1;
  double best_fill = fill(1);
  const int lim = std::min(max_splits, num_k / 8);
  for (int s = 2; s <= lim && best_fill < 0.93; ++s) {
    const double f = fill(s);
    if (f > best_fill + 1e-9) {
      best = s;
      best_fill = f;
    }
  }
  return best;
}

namespace {
__global__ void __launch_bounds__(256) splitk_reduce_kernel(int M, int N, int splits,
                                                            const float* __restrict__ part,
                                                            int64_t split_stride, int64_t ldp,
                                                            bf16* __restrict__ out, int64_t ldo) {
  const int nv = N / 8;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)M * nv) return;
  const int m = (int)(i / nv), c = (int)(i % nv) * 8;
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const float* pp = part + (int64_t)m * ldp + c;
  for (int s = 0; s < splits; ++s) {
    const float4 x = *reinterpret_cast<const float4*>(pp);
    const float4 y = *reinterpret_cast<const float4*>(pp + 4);
    a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
    a[4] += y.x; a[5] += y.y; a[6] += y.z; a[7] += y.w;
    pp += split_stride;
  }
  store8(out + (int64_t)m * ldo + c, a);
}
}  // namespace

mgb_status splitk_reduce_launch(int M, int N, int splits, const float* part, int64_t split_stride,
                                int64_t ldp, void* out, int64_t ldo, cudaStream_t st) {
  if (M < 0 || N < 0 || splits < 1 || N % 8 || ldp % 4 || ldo % 8 || split_stride % 4)
    return MGB_ERR_INVALID_ARG;
  const int64_t n = (int64_t)M * (N / 8);
  if (n == 0) return MGB_OK;
  LaunchScope scope(PROF_SPLITK_REDUCE, st);
  splitk_reduce_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(M, N, splits, part, split_stride,
                                                                    ldp, static_cast<bf16*>(out), ldo);
  return cudaGetLastError() == cudaSuccess ? MGB_OK : MGB_ERR_CUDA;
}

int device_sm_count() {
  static int sms[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) dev = 0;
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
    sms[dev] = n;
  }
  return sms[dev];
}

}  // namespace mgb
