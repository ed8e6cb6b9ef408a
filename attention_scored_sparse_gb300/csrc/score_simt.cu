// Window scoring, CUDA-core path (any D <= 128, bf16 or fp32).
//
// SparseEngine "How it works" (SnapKV / H2O scores from the attention of the
// window queries) and KARA Method 1 (bidirectional window scoring):
//     s[b, g, j] = sum_{h in g} sum_{q in window} softmax_j(q . k_j / sqrt(D))
//
// The softmax normaliser of a row is needed before its column can be summed,
// so scoring takes two sweeps over the keys:
//   pass 1  per (row tile, key split): running base-2 max / sum of each row;
//   lse     per row: combine the splits into lse2 = max + log2(sum);
//   pass 2  per key tile: recompute the logits of every row tile and sum
//           exp2(t - lse2) down the columns -- each CTA owns its columns, so
//           the column sums need no atomics and are deterministic.
// Rows of a group are ordered (window query, head in group).  This path is
// the fp32 kernel (tensor-core TF32 would miss fp32 accuracy) and the
// reference shape-coverage kernel for bf16; bf16 with D = 128 runs on the
// tcgen05 kernels.
#include "se_common.cuh"

namespace se {

struct ScoreArgs {
  se_paged_kv kv;
  const void* q_win;
  int w;
  const int32_t* q_pos;
  const int32_t* attn_lo;
  const int32_t* attn_hi;
  const int32_t* out_lo;
  const int32_t* out_hi;
  int causal;
  int accumulate;
  int n_max;
  float* scores;
  int64_t scores_stride;
  float* part;     // [B*Hkv][rows][n_splits][2]
  float* lse;      // [B*Hkv][rows]
  int n_splits;
  int split_keys;
};

template <typename T>
SE_DEV float to_f(T x) {
  if constexpr (sizeof(T) == 2) return __bfloat162float(x);
  else return x;
}

SE_DEV float ex2f_acc(float x) { return exp2f(x); }

constexpr int kTile = 32;

// Loads a tile of 32 rows of Q (scaled) and 32 keys into padded smem.
template <typename T>
SE_DEV void load_q_tile(const ScoreArgs& a, int b, int g, int r0, int rows, float* sq, int D) {
  const int G = a.kv.Hq / a.kv.Hkv;
  const float scale = kLog2e * rsqrtf((float)D);
  const T* q = static_cast<const T*>(a.q_win);
  for (int x = threadIdx.x; x < kTile * D; x += blockDim.x) {
    const int r = x / D, d = x % D;
    float v = 0.f;
    if (r0 + r < rows) {
      const int qi = (r0 + r) / G, j = (r0 + r) % G;
      v = to_f(q[(((int64_t)b * a.w + qi) * a.kv.Hq + g * G + j) * D + d]) * scale;
    }
    sq[r * (D + 1) + d] = v;
  }
}

template <typename T>
SE_DEV void load_k_tile(const ScoreArgs& a, int b, int g, int lo, int k0, int n, float* sk,
                        int* spos, int D) {
  const int P = a.kv.page_size;
  const T* kp = static_cast<const T*>(a.kv.k_pool);
  const int32_t* bt = a.kv.block_table + (int64_t)b * a.kv.max_pages_per_seq;
  const int64_t smax = (int64_t)a.kv.max_pages_per_seq * P;
  for (int x = threadIdx.x; x < kTile * D; x += blockDim.x) {
    const int kk = x / D, d = x % D;
    float v = 0.f;
    if (k0 + kk < n) {
      const int s = lo + k0 + kk;
      const int page = bt[s / P];
      if (page >= 0 && page < a.kv.num_pages)
        v = to_f(kp[(((int64_t)page * a.kv.Hkv + g) * P + s % P) * D + d]);
      else if (d == 0)
        set_status(a.kv.status, SE_ERR_BOUNDS);
    }
    sk[kk * (D + 1) + d] = v;
  }
  for (int kk = threadIdx.x; kk < kTile; kk += blockDim.x)
    spos[kk] = (k0 + kk < n) ? a.kv.slot_map[((int64_t)b * a.kv.Hkv + g) * smax + lo + k0 + kk]
                             : 0x7fffffff;
}

// grid: (row tiles, n_splits, B*Hkv), 256 threads: thread = (row tid/8, keys tid%8 + 8i)
template <typename T>
__global__ void __launch_bounds__(256) score_stats_simt(ScoreArgs a, int D) {
  pdl_enter();
  extern __shared__ float smem[];
  float* sq = smem;                          // [32][D+1]
  float* sk = sq + kTile * (D + 1);          // [32][D+1]
  int* spos = reinterpret_cast<int*>(sk + kTile * (D + 1));
  const int bg = blockIdx.z, b = bg / a.kv.Hkv, g = bg % a.kv.Hkv;
  const int G = a.kv.Hq / a.kv.Hkv;
  const int rows = a.w * G;
  const int r0 = blockIdx.x * kTile;
  const int lo = a.attn_lo[b];
  int n = a.attn_hi[b] - lo;
  if (lo < 0 || n > a.n_max || (int64_t)(lo + n) > (int64_t)a.kv.max_pages_per_seq * a.kv.page_size) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) set_status(a.kv.status, SE_ERR_BOUNDS);
    n = 0;
  }
  const int kb = blockIdx.y * a.split_keys, ke = min(kb + a.split_keys, n);
  const int r = threadIdx.x / 8, kc = threadIdx.x % 8;
  const int qpos = (r0 + r < rows) ? a.q_pos[(int64_t)b * a.w + (r0 + r) / G] : 0;
  load_q_tile<T>(a, b, g, r0, rows, sq, D);
  float m = -INFINITY, l = 0.f;
  for (int k0 = kb; k0 < ke; k0 += kTile) {
    __syncthreads();
    load_k_tile<T>(a, b, g, lo, k0, ke, sk, spos, D);
    __syncthreads();
    float t[4] = {0.f, 0.f, 0.f, 0.f};
    for (int d = 0; d < D; ++d) {
      const float qv = sq[r * (D + 1) + d];
#pragma unroll
      for (int i = 0; i < 4; ++i) t[i] = fmaf(qv, sk[(kc + 8 * i) * (D + 1) + d], t[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int kk = kc + 8 * i;
      const bool vis = (k0 + kk < ke) && (!a.causal || spos[kk] <= qpos);
      if (vis) {
        const float mn = fmaxf(m, t[i]);
        l = l * ex2f_acc(m - mn) + ex2f_acc(t[i] - mn);
        m = mn;
      }
    }
  }
  // merge the 8 threads of a row
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float l2 = __shfl_xor_sync(0xffffffffu, l, o);
    const float mn = fmaxf(m, m2);
    if (mn != -INFINITY) {
      l = l * ex2f_acc(m - mn) + l2 * ex2f_acc(m2 - mn);
      m = mn;
    }
  }
  if (kc == 0 && r0 + r < rows) {
    float* p = a.part + (((int64_t)bg * rows + r0 + r) * a.n_splits + blockIdx.y) * 2;
    p[0] = m;
    p[1] = l;
  }
}

// lse2 per row from the split partials.  grid: (cdiv(rows,256), B*Hkv)
__global__ void score_lse_kernel(ScoreArgs a) {
  pdl_enter();
  const int bg = blockIdx.y;
  const int G = a.kv.Hq / a.kv.Hkv;
  const int rows = a.w * G;
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= rows) return;
  const float* p = a.part + ((int64_t)bg * rows + r) * a.n_splits * 2;
  float M = -INFINITY;
  for (int s = 0; s < a.n_splits; ++s) M = fmaxf(M, p[2 * s]);
  float L = 0.f;
  if (M != -INFINITY)
    for (int s = 0; s < a.n_splits; ++s) L += p[2 * s + 1] * exp2f(p[2 * s] - M);
  a.lse[(int64_t)bg * rows + r] = (L > 0.f) ? M + log2f(L) : INFINITY;
}

// grid: (key tiles of the output range, 1, B*Hkv), 256 threads:
// thread = (key tid%32, rows tid/32 + 8i)
template <typename T>
__global__ void __launch_bounds__(256) score_colsum_simt(ScoreArgs a, int D) {
  pdl_enter();
  extern __shared__ float smem[];
  float* sq = smem;
  float* sk = sq + kTile * (D + 1);
  int* spos = reinterpret_cast<int*>(sk + kTile * (D + 1));
  __shared__ float s_lse[kTile];
  __shared__ int s_qpos[kTile];
  __shared__ float s_red[8][kTile];
  const int bg = blockIdx.z, b = bg / a.kv.Hkv, g = bg % a.kv.Hkv;
  const int G = a.kv.Hq / a.kv.Hkv;
  const int rows = a.w * G;
  const int lo = a.attn_lo[b], n = a.attn_hi[b] - lo;
  const int olo = a.out_lo[b] - lo, ohi = a.out_hi[b] - lo;
  const int k0 = olo + blockIdx.x * kTile;
  if (k0 >= ohi) return;
  if (lo < 0 || n > a.n_max || olo < 0 || ohi > n || lo + ohi > a.scores_stride ||
      (int64_t)(lo + n) > (int64_t)a.kv.max_pages_per_seq * a.kv.page_size) {
    if (threadIdx.x == 0) set_status(a.kv.status, SE_ERR_BOUNDS);
    return;
  }
  const int kk = threadIdx.x % kTile, rs = threadIdx.x / kTile;
  load_k_tile<T>(a, b, g, lo, k0, min(ohi, n), sk, spos, D);
  float colsum = 0.f;
  for (int r0 = 0; r0 < rows; r0 += kTile) {
    __syncthreads();
    load_q_tile<T>(a, b, g, r0, rows, sq, D);
    for (int x = threadIdx.x; x < kTile; x += blockDim.x) {
      s_lse[x] = (r0 + x < rows) ? a.lse[(int64_t)bg * rows + r0 + x] : INFINITY;
      s_qpos[x] = (r0 + x < rows) ? a.q_pos[(int64_t)b * a.w + (r0 + x) / G] : 0;
    }
    __syncthreads();
    float t[4] = {0.f, 0.f, 0.f, 0.f};
    for (int d = 0; d < D; ++d) {
      const float kv = sk[kk * (D + 1) + d];
#pragma unroll
      for (int i = 0; i < 4; ++i) t[i] = fmaf(sq[(rs + 8 * i) * (D + 1) + d], kv, t[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int rr = rs + 8 * i;
      const bool vis = (r0 + rr < rows) && (!a.causal || spos[kk] <= s_qpos[rr]) &&
                       s_lse[rr] != INFINITY;
      if (vis) colsum += ex2f_acc(t[i] - s_lse[rr]);
    }
  }
  s_red[rs][kk] = colsum;
  __syncthreads();
  if (rs == 0 && k0 + kk < ohi) {
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) v += s_red[i][kk];
    float* out = a.scores + (int64_t)bg * a.scores_stride + lo + k0 + kk;
    *out = a.accumulate ? *out + v : v;
  }
}

size_t score_simt_ws(const se_paged_kv* kv, int w, int n_max, int* n_splits, int* split_keys) {
  const int G = kv->Hq / kv->Hkv;
  const int rows = w * G;
  const int sk = 256;
  const int ns = cdiv(max(n_max, 1), sk);
  if (n_splits) *n_splits = ns;
  if (split_keys) *split_keys = sk;
  WsCarver c(nullptr);
  c.take<float>((size_t)kv->B * kv->Hkv * rows * ns * 2);
  c.take<float>((size_t)kv->B * kv->Hkv * rows);
  return c.bytes();
}

se_status launch_score_simt(ScoreArgs a, void* ws, cudaStream_t st) {
  const se_paged_kv* kv = &a.kv;
  const int G = kv->Hq / kv->Hkv;
  const int rows = a.w * G;
  score_simt_ws(kv, a.w, a.n_max, &a.n_splits, &a.split_keys);
  WsCarver c(ws);
  a.part = c.take<float>((size_t)kv->B * kv->Hkv * rows * a.n_splits * 2);
  a.lse = c.take<float>((size_t)kv->B * kv->Hkv * rows);
  const int D = kv->D;
  const size_t smem = (size_t)(2 * kTile * (D + 1) + kTile) * sizeof(float);
  dim3 g1(cdiv(rows, kTile), a.n_splits, kv->B * kv->Hkv);
  dim3 g2(cdiv(a.n_max, kTile), 1, kv->B * kv->Hkv);
  if (kv->dtype == SE_BF16) {
    se_launch(score_stats_simt<__nv_bfloat16>, g1, 256, smem, st, a, D);
    se_launch(score_lse_kernel, dim3(cdiv(rows, 256), kv->B * kv->Hkv), 256, 0, st, a);
    se_launch(score_colsum_simt<__nv_bfloat16>, g2, 256, smem, st, a, D);
  } else {
    se_launch(score_stats_simt<float>, g1, 256, smem, st, a, D);
    se_launch(score_lse_kernel, dim3(cdiv(rows, 256), kv->B * kv->Hkv), 256, 0, st, a);
    se_launch(score_colsum_simt<float>, g2, 256, smem, st, a, D);
  }
  return SE_OK;
}

bool score_tc_supported(const se_paged_kv* kv);
size_t score_tc_ws(const se_paged_kv* kv, int w, int n_max);
se_status launch_score_tc(const se_paged_kv* kv, const void* q_win, int w, const int32_t* q_pos,
                          const int32_t* attn_lo, const int32_t* attn_hi, const int32_t* out_lo,
                          const int32_t* out_hi, int causal, int accumulate, int n_max,
                          float* scores, int64_t scores_stride, void* ws, cudaStream_t st,
                          int one_launch);

}  // namespace se

using namespace se;

// bf16 with D = 128 runs on the tcgen05 kernels; everything else (fp32, D = 64)
// on the CUDA-core kernels above.
extern "C" size_t se_score_window_workspace_size(const se_paged_kv* kv, int32_t w, int32_t n_max) {
  if (kv == nullptr || w < 0 || n_max < 0) return 0;
  if (score_tc_supported(kv)) return score_tc_ws(kv, w, n_max);
  return score_simt_ws(kv, w, n_max, nullptr, nullptr);
}

static se_status score_window_impl(const se_paged_kv* kv, const void* q_win, int32_t w,
                                   const int32_t* q_pos, const int32_t* attn_lo,
                                   const int32_t* attn_hi, const int32_t* out_lo,
                                   const int32_t* out_hi, int32_t causal, int32_t accumulate,
                                   int32_t n_max, float* scores, int64_t scores_stride,
                                   void* workspace, size_t workspace_bytes, void* stream,
                                   int one_launch) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (q_win == nullptr || q_pos == nullptr || attn_lo == nullptr || attn_hi == nullptr ||
      out_lo == nullptr || out_hi == nullptr || scores == nullptr || workspace == nullptr ||
      w < 1 || n_max < 1)
    return SE_ERR_INVALID_ARG;
  if (workspace_bytes < se_score_window_workspace_size(kv, w, n_max)) return SE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (score_tc_supported(kv)) {
    s = launch_score_tc(kv, q_win, w, q_pos, attn_lo, attn_hi, out_lo, out_hi, causal, accumulate,
                        n_max, scores, scores_stride, workspace, st, one_launch);
  } else if (one_launch) {
    return SE_ERR_UNSUPPORTED;
  } else {
    ScoreArgs a{*kv, q_win, w, q_pos, attn_lo, attn_hi, out_lo, out_hi, causal, accumulate,
                n_max, scores, scores_stride, nullptr, nullptr, 0, 0};
    s = launch_score_simt(a, workspace, st);
  }
  if (s != SE_OK) return s;
  return se_last_launch_status();
}

extern "C" se_status se_score_window(const se_paged_kv* kv, const void* q_win, int32_t w,
                                     const int32_t* q_pos, const int32_t* attn_lo,
                                     const int32_t* attn_hi, const int32_t* out_lo,
                                     const int32_t* out_hi, int32_t causal, int32_t accumulate,
                                     int32_t n_max, float* scores, int64_t scores_stride,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  return score_window_impl(kv, q_win, w, q_pos, attn_lo, attn_hi, out_lo, out_hi, causal,
                           accumulate, n_max, scores, scores_stride, workspace, workspace_bytes,
                           stream, 0);
}

extern "C" se_status se_score_window_one_launch(const se_paged_kv* kv, const void* q_win, int32_t w,
                                                const int32_t* q_pos, const int32_t* attn_lo,
                                                const int32_t* attn_hi, const int32_t* out_lo,
                                                const int32_t* out_hi, int32_t causal,
                                                int32_t accumulate, int32_t n_max, float* scores,
                                                int64_t scores_stride, void* workspace,
                                                size_t workspace_bytes, void* stream) {
  return score_window_impl(kv, q_win, w, q_pos, attn_lo, attn_hi, out_lo, out_hi, causal,
                           accumulate, n_max, scores, scores_stride, workspace, workspace_bytes,
                           stream, 1);
}
