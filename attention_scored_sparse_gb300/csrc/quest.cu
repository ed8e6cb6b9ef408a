// Quest page metadata and query-dependent page selection.
//
// SparseEngine "How it works" (build_decode_selection performs Quest's
// query-dependent page selection; metadata persists beside the KV state) and
// "How it differs" (Quest keeps the full KV history).  The bound per page p
// and KV group g is sum_{h in g} sum_d max(q_hd * kmax_pd, q_hd * kmin_pd).
//
// Both kernels stream HBM: the metadata build reads every resident key once
// (16-byte loads, one CTA per page, 16 threads per head row); the bound
// kernel reads 2*D elements per (page, group) with one half-warp per page and
// the group's queries held in registers, writes one float per page, and the
// shared block radix top-k then picks the pages.
#include "tc_primitives.cuh"

namespace se {

se_status launch_topk_select_pages(int B, int Hkv, const float* U, int64_t stride,
                                   const int32_t* cand_lo, const int32_t* cand_hi,
                                   const int32_t* force_lo,
                                   const int32_t* force_hi, int32_t* out, int32_t out_stride,
                                   int32_t* n_sel, int32_t* status, int top, int n_max,
                                   cudaStream_t st);

// grid: (blocks of a sequence, B); threads: Hkv * (row_bytes/16) <= 1024
template <typename T>
__global__ void quest_meta_kernel(se_paged_kv kv, T* kmin, T* kmax) {
  pdl_enter();
  const int blk = blockIdx.x, b = blockIdx.y;
  const int P = kv.page_size;
  const int ctx = kv.ctx_len[b];
  if (blk * P >= ctx) return;
  const int rows = min(P, ctx - blk * P);
  const int page = kv.block_table[(int64_t)b * kv.max_pages_per_seq + blk];
  constexpr int EPC = 16 / sizeof(T);  // elements per 16-byte chunk
  const int chunks = kv.D / EPC;
  const int t = threadIdx.x;
  if (t >= kv.Hkv * chunks) return;
  const int h = t / chunks, c = t % chunks;
  const T* base = static_cast<const T*>(kv.k_pool) + (((int64_t)page * kv.Hkv + h) * P) * kv.D + c * EPC;
  float mn[EPC], mx[EPC];
#pragma unroll
  for (int i = 0; i < EPC; ++i) { mn[i] = INFINITY; mx[i] = -INFINITY; }
  for (int r = 0; r < rows; ++r) {
    const uint4 u = ldg_nc_v4(base + (int64_t)r * kv.D);
    float f[EPC];
    if constexpr (sizeof(T) == 2) {
      unpack8_bf16(u, f);
    } else {
      f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
      f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    }
#pragma unroll
    for (int i = 0; i < EPC; ++i) { mn[i] = fminf(mn[i], f[i]); mx[i] = fmaxf(mx[i], f[i]); }
  }
  const int64_t o = ((int64_t)page * kv.Hkv + h) * kv.D + c * EPC;
#pragma unroll
  for (int i = 0; i < EPC; ++i) {
    if constexpr (sizeof(T) == 2) {
      kmin[o + i] = __float2bfloat16_rn(mn[i]);  // exact: a bf16 value
      kmax[o + i] = __float2bfloat16_rn(mx[i]);
    } else {
      kmin[o + i] = mn[i];
      kmax[o + i] = mx[i];
    }
  }
}

// Candidate and forced ranges of sequence b's top-k: candidates are the full
// blocks [0, nb - 1), the current block nb - 1 is forced.  A sequence longer
// than the bound buffer is reported and selected among its first max_blocks.
struct QuestRanges {
  int32_t* cand_lo;
  int32_t* cand_hi;
  int32_t* flo;
  int32_t* fhi;
};

SE_DEV void write_ranges(const QuestRanges& r, int32_t* status, int b, int nb, int max_blocks) {
  if (nb > max_blocks) {
    set_status(status, SE_ERR_BOUNDS);
    nb = max_blocks;
  }
  r.cand_lo[b] = 0;
  r.cand_hi[b] = max(nb - 1, 0);
  r.flo[b] = max(nb - 1, 0);
  r.fhi[b] = nb;
}

// Page bound U for every full block; CTA (0, 0, b) also writes sequence b's
// ranges.  grid: (cdiv(max_blocks, kBoundPages * 16 / hpc), Hkv / hpc, B),
// 256 threads = 8 warps; warp w serves KV head blockIdx.y * hpc + w % hpc
// (hpc = heads per CTA, min(Hkv, 8)), so the warps of a CTA read the kmin /
// kmax rows of all hpc heads of a page together: hpc x 256 contiguous bytes
// each, the heads of a physical page being adjacent in the metadata.  Each
// half-warp takes kBoundPages blocks (16 / hpc apart, so a warp's
// block-table reads are contiguous) with all their loads in flight together.
// The block-table reads do not wait for ctx_len (only the mask does).
// D = 128 bf16: lane t of the half-warp owns dims [8t, 8t+8).
//
// The sum over the group's heads is taken on the query side: with
// kmax >= kmin, max(q kmax, q kmin) = max(q, 0) kmax + min(q, 0) kmin, so
// U = sum_d (sum_h max(q_hd, 0)) kmax_d + (sum_h min(q_hd, 0)) kmin_d --
// two FMAs per dimension whatever the group size, and 16 query registers.
constexpr int kBoundPages = 8;   // blocks per half-warp

template <int G>
__global__ void __launch_bounds__(256) quest_bound_bf16_kernel(se_paged_kv kv,
                                                               const __nv_bfloat16* __restrict__ kmin,
                                                               const __nv_bfloat16* __restrict__ kmax,
                                                               const __nv_bfloat16* __restrict__ q,
                                                               float* __restrict__ U,
                                                               int64_t u_stride, int hpc,
                                                               QuestRanges rg) {
  pdl_enter();
  const int b = blockIdx.z;
  const int P = kv.page_size;
  const int warp = threadIdx.x >> 5, t = threadIdx.x & 15;
  const int g = blockIdx.y * hpc + warp % hpc;
  const int rows = 16 / hpc;                                  // half-warps per head
  const int hi = (warp / hpc) * 2 + ((threadIdx.x >> 4) & 1);  // this half-warp among them
  const int ctx = kv.ctx_len[b];
  const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
  int blk[kBoundPages], page[kBoundPages];
#pragma unroll
  for (int u = 0; u < kBoundPages; ++u) {
    blk[u] = blockIdx.x * rows * kBoundPages + u * rows + hi;
    page[u] = blk[u] < u_stride ? bt[blk[u]] : -1;
  }
  float qp[8], qn[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    qp[i] = 0.f;
    qn[i] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const uint4 u = ldg_nc_v4(q + ((int64_t)b * kv.Hq + g * G + j) * kv.D + t * 8);
    float qv[8];
    unpack8_bf16(u, qv);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      qp[i] += fmaxf(qv[i], 0.f);
      qn[i] += fminf(qv[i], 0.f);
    }
  }
  const int nb = cdiv(ctx, P);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    write_ranges(rg, kv.status, b, nb, (int)u_stride);
  bool act[kBoundPages];
  uint4 mnr[kBoundPages], mxr[kBoundPages];
#pragma unroll
  for (int u = 0; u < kBoundPages; ++u) {
    act[u] = blk[u] < nb - 1 && page[u] >= 0 && page[u] < kv.num_pages;
    if (act[u]) {
      const int64_t o = ((int64_t)page[u] * kv.Hkv + g) * kv.D + t * 8;
      mnr[u] = ldg_nc_v4(kmin + o);
      mxr[u] = ldg_nc_v4(kmax + o);
    }
  }
#pragma unroll
  for (int u = 0; u < kBoundPages; ++u) {
    float acc = 0.f;
    if (act[u]) {
      float mn[8], mx[8];
      unpack8_bf16(mnr[u], mn);
      unpack8_bf16(mxr[u], mx);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc = fmaf(qn[i], mn[i], fmaf(qp[i], mx[i], acc));
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (act[u] && t == 0) U[((int64_t)b * kv.Hkv + g) * u_stride + blk[u]] = acc;
  }
}

// Page bound over a ring of bulk-copied stages (bf16, D = 128): the same
// bounds as quest_bound_bf16_kernel, with each CTA keeping copies in flight
// across many pages.  grid: (cdiv(max_blocks, L), Hkv / hpc, B), 256
// threads, dynamic smem kQbStages x 32 KB.  CTA (x, y, b) takes the blocks
// [L x, L (x + 1)) of sequence b (L a multiple of SB = 64 / hpc blocks, at
// most eight stages) for heads [y hpc, (y + 1) hpc).  Warp 0 copies, per block, the kmin
// rows of the hpc heads (hpc x 256 contiguous bytes) and their kmax rows into
// a stage; two stages are in flight while the CTA computes a third.
// Half-warp h serves head y hpc + h % hpc for the whole launch (its folded
// query in 16 registers) and in round r of a stage the block (16 r + h) /
// hpc.  CTA (0, 0, b) also writes sequence b's ranges.  Every wait is
// bounded; one that runs out sets SE_ERR_TIMEOUT and the CTA drains its
// copies and leaves.
constexpr int kQbStages = 3;
constexpr int kQbStageBytes = 32768;       // kmin half, then kmax half
constexpr int kQbStagesPerCta = 8;
constexpr int kQbMaxBlocks = kQbStagesPerCta * 64;

template <int G>
__global__ void __launch_bounds__(256, 2) quest_bound_ring_kernel(
    se_paged_kv kv, const __nv_bfloat16* __restrict__ kmin, const __nv_bfloat16* __restrict__ kmax,
    const __nv_bfloat16* __restrict__ q, float* __restrict__ U, int64_t u_stride, int hpc, int L,
    QuestRanges rg) {
  extern __shared__ __align__(128) uint8_t qb_smem[];
  __shared__ uint64_t full[kQbStages], empty[kQbStages];
  __shared__ int32_t s_page[kQbMaxBlocks];
  __shared__ int s_abort;
  constexpr uint64_t kLimit = 2000000000ull;
  const int b = blockIdx.z;
  const int P = kv.page_size;
  const int SB = 64 / hpc;                    // blocks per stage
  const int x0 = blockIdx.x * L;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = threadIdx.x >> 4, t = threadIdx.x & 15;
  const int hh = h % hpc, g = blockIdx.y * hpc + hh;
  const uint32_t row_bytes = (uint32_t)hpc * 256u;   // hpc heads x 128 bf16
  uint8_t* stages = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(qb_smem) + 127) & ~uintptr_t(127));
  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < kQbStages; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 8);
    }
    tc::fence_barrier_init();
  }
  pdl_enter();
  const int ctx = kv.ctx_len[b];
  const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
  // the CTA's block-table entries (these reads do not wait for ctx_len)
  for (int i = threadIdx.x; i < L; i += blockDim.x)
    s_page[i] = x0 + i < u_stride ? bt[x0 + i] : -1;
  float qp[8], qn[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    qp[i] = 0.f;
    qn[i] = 0.f;
  }
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const uint4 u = ldg_nc_v4(q + ((int64_t)b * kv.Hq + g * G + j) * kv.D + t * 8);
    float qv[8];
    unpack8_bf16(u, qv);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      qp[i] += fmaxf(qv[i], 0.f);
      qn[i] += fminf(qv[i], 0.f);
    }
  }
  const int nb = cdiv(ctx, P);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    write_ranges(rg, kv.status, b, nb, (int)u_stride);
  __syncthreads();
  // full blocks [0, nb - 1) of this CTA, as a count from x0
  const int n_blocks = max(min(min(nb - 1, (int)u_stride) - x0, L), 0);
  const int n_stages = cdiv(n_blocks, SB);
  const char* kmn = reinterpret_cast<const char*>(kmin);
  const char* kmx = reinterpret_cast<const char*>(kmax);
  const int64_t head0 = (int64_t)blockIdx.y * hpc * 256;   // byte offset of head y hpc in a page's rows

  // copies of stage n: block j of the stage by lane j (and j + 32)
  auto issue = [&](int n) {
    uint8_t* st = stages + (n % kQbStages) * kQbStageBytes;
    for (int j = lane; j < SB; j += 32) {
      const int i = n * SB + j;
      const int page = i < n_blocks ? s_page[i] : -1;
      if (page >= 0 && page < kv.num_pages) {
        const int64_t src = (int64_t)page * kv.Hkv * 256 + head0;
        tc::bulk_g2s(st + j * row_bytes, kmn + src, row_bytes, &full[n % kQbStages]);
        tc::bulk_g2s(st + kQbStageBytes / 2 + j * row_bytes, kmx + src, row_bytes,
                     &full[n % kQbStages]);
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&full[n % kQbStages]);
  };

  int issued = 0;
  if (warp == 0)
    for (; issued < min(kQbStages - 1, n_stages); ++issued) issue(issued);
  for (int n = 0; n < n_stages; ++n) {
    if (warp == 0 && issued < n_stages) {
      // refill the buffer released in the previous iteration
      const int m = issued;
      const bool ok = m < kQbStages ||
                      tc::mbar_wait(&empty[m % kQbStages], ((m / kQbStages) - 1) & 1, kLimit);
      if (__all_sync(0xffffffffu, ok)) {
        issue(m);
        ++issued;
      } else if (lane == 0) {
        set_status(kv.status, SE_ERR_TIMEOUT);
        atomicExch(&s_abort, 1);
      }
    }
    const bool landed = tc::mbar_wait(&full[n % kQbStages], (n / kQbStages) & 1, kLimit);
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) {
        set_status(kv.status, SE_ERR_TIMEOUT);
        atomicExch(&s_abort, 1);
      }
      break;
    }
    const uint8_t* st = stages + (n % kQbStages) * kQbStageBytes;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int j = (16 * r + h) / hpc;          // block of the stage
      const int i = n * SB + j;
      const int page = i < n_blocks ? s_page[i] : -1;
      const bool act = page >= 0 && page < kv.num_pages;
      float acc = 0.f;
      if (act) {
        const int off = j * row_bytes + hh * 256 + t * 16;
        float mn[8], mx[8];
        unpack8_bf16(*reinterpret_cast<const uint4*>(st + off), mn);
        unpack8_bf16(*reinterpret_cast<const uint4*>(st + kQbStageBytes / 2 + off), mx);
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = fmaf(qn[e], mn[e], fmaf(qp[e], mx[e], acc));
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (act && t == 0) U[((int64_t)b * kv.Hkv + g) * u_stride + x0 + i] = acc;
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&empty[n % kQbStages]);
  }
  // after a timeout, copies of issued stages may still be in flight
  if (warp == 0 && lane == 0)
    for (int m = max(0, issued - kQbStages); m < issued; ++m)
      tc::mbar_wait(&full[m % kQbStages], (m / kQbStages) & 1, kLimit);
}

// Generic bound (any D, fp32 or bf16): one thread per (block, group); CTA
// (0, 0, b) also writes sequence b's ranges.
template <typename T>
__global__ void quest_bound_generic_kernel(se_paged_kv kv, const T* kmin, const T* kmax,
                                           const T* q, float* U, int64_t u_stride, QuestRanges rg) {
  pdl_enter();
  const int g = blockIdx.y, b = blockIdx.z;
  const int blk = blockIdx.x * blockDim.x + threadIdx.x;
  const int nb = cdiv(kv.ctx_len[b], kv.page_size);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
    write_ranges(rg, kv.status, b, nb, (int)u_stride);
  if (blk >= nb - 1 || blk >= u_stride) return;
  const int G = kv.Hq / kv.Hkv;
  const int page = kv.block_table[(int64_t)b * kv.max_pages_per_seq + blk];
  if (page < 0 || page >= kv.num_pages) return;
  const int64_t o = ((int64_t)page * kv.Hkv + g) * kv.D;
  float acc = 0.f;
  for (int j = 0; j < G; ++j) {
    const T* qh = q + ((int64_t)b * kv.Hq + g * G + j) * kv.D;
    float part = 0.f;
    for (int d = 0; d < kv.D; ++d) {
      const float x = (float)qh[d];
      part += fmaxf(x * (float)kmax[o + d], x * (float)kmin[o + d]);
    }
    acc += part;
  }
  U[((int64_t)b * kv.Hkv + g) * u_stride + blk] = acc;
}

struct QuestWs {
  float* U;
  int32_t* cand_lo;
  int32_t* cand_hi;
  int32_t* flo;
  int32_t* fhi;
  int64_t u_stride;
};

static QuestWs carve_quest(const se_paged_kv* kv, int32_t max_blocks, void* ws, size_t* bytes) {
  WsCarver c(ws);
  QuestWs w;
  w.u_stride = max_blocks;
  w.U = c.take<float>((size_t)kv->B * kv->Hkv * max_blocks);
  w.cand_lo = c.take<int32_t>(kv->B);
  w.cand_hi = c.take<int32_t>(kv->B);
  w.flo = c.take<int32_t>(kv->B);
  w.fhi = c.take<int32_t>(kv->B);
  *bytes = c.bytes();
  return w;
}

// The ring kernel's shared memory above 48 KB, allowed once per device and
// group size; false where the device refuses it (the bound then runs in the
// register kernel).
static bool ring_ready(int G) {
  const int smem = kQbStages * kQbStageBytes + 128;
  static std::atomic<uint64_t> a1{0}, a2{0}, a4{0}, a8{0};
  switch (G) {
    case 1: return allow_smem(reinterpret_cast<const void*>(&quest_bound_ring_kernel<1>), smem, a1);
    case 2: return allow_smem(reinterpret_cast<const void*>(&quest_bound_ring_kernel<2>), smem, a2);
    case 4: return allow_smem(reinterpret_cast<const void*>(&quest_bound_ring_kernel<4>), smem, a4);
    case 8: return allow_smem(reinterpret_cast<const void*>(&quest_bound_ring_kernel<8>), smem, a8);
    default: return false;
  }
}

}  // namespace se

using namespace se;

extern "C" se_status se_quest_build_meta(const se_paged_kv* kv, void* kmin, void* kmax,
                                         void* stream) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (kmin == nullptr || kmax == nullptr) return SE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int threads = kv->Hkv * kv->D * (int)elem_size(kv->dtype) / 16;
  if (threads > 1024) return SE_ERR_UNSUPPORTED;
  dim3 grid(kv->max_pages_per_seq, kv->B);
  if (kv->dtype == SE_BF16)
    se_launch(quest_meta_kernel<__nv_bfloat16>, grid, threads, 0, st,
        *kv, static_cast<__nv_bfloat16*>(kmin), static_cast<__nv_bfloat16*>(kmax));
  else
    se_launch(quest_meta_kernel<float>, grid, threads, 0, st, *kv, static_cast<float*>(kmin),
                                                       static_cast<float*>(kmax));
  return se_last_launch_status();
}

extern "C" size_t se_quest_page_select_workspace_size(const se_paged_kv* kv, int32_t max_blocks) {
  if (kv == nullptr) return 0;
  size_t b = 0;
  carve_quest(kv, max_blocks, nullptr, &b);
  return b;
}


extern "C" se_status se_quest_page_select(const se_paged_kv* kv, const void* kmin,
                                          const void* kmax, const void* q, int32_t top_pages,
                                          int32_t max_blocks, int32_t* page_idx, int32_t* n_sel,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (kmin == nullptr || kmax == nullptr || q == nullptr || page_idx == nullptr ||
      workspace == nullptr || top_pages < 0 || max_blocks < 1 ||
      max_blocks > kv->max_pages_per_seq)
    return SE_ERR_INVALID_ARG;
  size_t need = 0;
  QuestWs w = carve_quest(kv, max_blocks, workspace, &need);
  if (workspace_bytes < need) return SE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int G = kv->Hq / kv->Hkv;
  const QuestRanges rg{w.cand_lo, w.cand_hi, w.flo, w.fhi};
  const int hpc = kv->Hkv % 8 == 0 ? 8 : (kv->Hkv < 8 && 8 % kv->Hkv == 0 ? kv->Hkv : 0);
  const bool bf16_128 = kv->dtype == SE_BF16 && kv->D == 128 && hpc > 0 &&
                        (G == 1 || G == 2 || G == 4 || G == 8);
  auto km = static_cast<const __nv_bfloat16*>(kmin);
  auto kx = static_cast<const __nv_bfloat16*>(kmax);
  auto qq = static_cast<const __nv_bfloat16*>(q);
  if (bf16_128 && ring_ready(G)) {
    // one even wave of two CTAs per SM where the blocks allow it: L blocks
    // per CTA, a multiple of a stage, at most eight stages
    const int SB = 64 / hpc;
    const int sets = kv->B * (kv->Hkv / hpc);
    const int nx0 = max(cdiv(2 * 152, sets), cdiv(max_blocks, kQbMaxBlocks));
    const int L = cdiv(cdiv(max_blocks, nx0), SB) * SB;
    const dim3 grid(cdiv(max_blocks, L), kv->Hkv / hpc, kv->B);
    const int smem = kQbStages * kQbStageBytes + 128;
    if (G == 1) se_launch(quest_bound_ring_kernel<1>, grid, 256, smem, st, *kv, km, kx, qq, w.U, w.u_stride, hpc, L, rg);
    if (G == 2) se_launch(quest_bound_ring_kernel<2>, grid, 256, smem, st, *kv, km, kx, qq, w.U, w.u_stride, hpc, L, rg);
    if (G == 4) se_launch(quest_bound_ring_kernel<4>, grid, 256, smem, st, *kv, km, kx, qq, w.U, w.u_stride, hpc, L, rg);
    if (G == 8) se_launch(quest_bound_ring_kernel<8>, grid, 256, smem, st, *kv, km, kx, qq, w.U, w.u_stride, hpc, L, rg);
  } else if (bf16_128) {
    const dim3 grid(cdiv(max_blocks, 16 / hpc * kBoundPages), kv->Hkv / hpc, kv->B);
    if (G == 1) se_launch(quest_bound_bf16_kernel<1>, grid, 256, 0, st, *kv, km, kx, qq, w.U, w.u_stride, hpc, rg);
    if (G == 2) se_launch(quest_bound_bf16_kernel<2>, grid, 256, 0, st, *kv, km, kx, qq, w.U, w.u_stride, hpc, rg);
    if (G == 4) se_launch(quest_bound_bf16_kernel<4>, grid, 256, 0, st, *kv, km, kx, qq, w.U, w.u_stride, hpc, rg);
    if (G == 8) se_launch(quest_bound_bf16_kernel<8>, grid, 256, 0, st, *kv, km, kx, qq, w.U, w.u_stride, hpc, rg);
  } else {
    dim3 g2(cdiv(max_blocks, 128), kv->Hkv, kv->B);
    if (kv->dtype == SE_BF16)
      se_launch(quest_bound_generic_kernel<__nv_bfloat16>, g2, 128, 0, st,
          *kv, static_cast<const __nv_bfloat16*>(kmin), static_cast<const __nv_bfloat16*>(kmax),
          static_cast<const __nv_bfloat16*>(q), w.U, w.u_stride, rg);
    else
      se_launch(quest_bound_generic_kernel<float>, g2, 128, 0, st,
          *kv, static_cast<const float*>(kmin), static_cast<const float*>(kmax),
          static_cast<const float*>(q), w.U, w.u_stride, rg);
  }
  s = launch_topk_select_pages(kv->B, kv->Hkv, w.U, w.u_stride, w.cand_lo, w.cand_hi, w.flo,
                               w.fhi, page_idx, top_pages + 1, n_sel, kv->status, top_pages,
                               max_blocks, st);
  if (s != SE_OK) return s;
  return se_last_launch_status();
}
