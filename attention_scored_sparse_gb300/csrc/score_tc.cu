// Window scoring on the 5th-generation tensor cores (bf16, D = 128).
//
// SparseEngine "How it works" (SnapKV / H2O: attention of the window queries
// over the cached keys) and KARA Method 1 (bidirectional window scoring):
//     s[b, g, j] = sum_{h in g} sum_{q in window} softmax_j(q . k_j / sqrt(D))
// Rows of a group are (window query, head in group); the softmax of a row is
// needed before its column can be summed, so there are two sweeps:
//
//   pass 1 (rowstats)  S = Q_rows K_tile^T with the 256 rows of a chunk on
//       TMEM lanes (two M=128 accumulators), N = 128 keys; each epilogue
//       thread owns one row and one 64-key half of every tile and keeps a
//       base-2 running max / sum over its CTA's key range.  Partials per
//       (key split, half) go to the workspace.
//   rowinfo            the splits merge into -lse2 per row (plus the row's
//       query position for causal masking): a CUDA-core kernel when the rows
//       span several chunks, pass 2's epilogue itself in the persistent form.
//   pass 2 (colsum)    S^T = K_tile Q_rows^T with the 128 keys of a tile on
//       TMEM lanes (M=128), N = 256 rows; each epilogue thread owns one key
//       and one 128-row half and sums exp2(t - lse2_r) over its rows in
//       registers; the two halves of a key meet once in shared memory.
//
// Both passes: one producer warp issues TMA loads (K pages as 16-row boxes
// gathered through the block table, 128-byte swizzle; Q via a 4-D map over
// [B][w][Hq][D]; key positions and row info as 1-D bulk copies), one warp
// issues tcgen05.mma from shared-memory descriptors into double-buffered TMEM
// accumulators, sixteen warps (four per SM sub-partition, so that exp2,
// FMA and TMEM-load latencies overlap) run the epilogue from tcgen05.ld.  Every
// mbarrier wait is bounded by %globaltimer: on expiry the CTA records
// SE_ERR_TIMEOUT, drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>

#include <algorithm>

#include "tc_primitives.cuh"

namespace se {

namespace {

constexpr int kD = 128;
constexpr int kKeyTile = 128;       // keys per tile (M of pass 2, N of pass 1)
constexpr int kRowChunk = 256;      // rows per chunk (2 x M=128 in pass 1, N of pass 2)
constexpr int kKTileBytes = kKeyTile * kD * 2;   // 32 KB
constexpr int kQChunkBytes = kRowChunk * kD * 2; // 64 KB
constexpr int kStages1 = 4;         // K-tile ring depth, pass 1
constexpr int kEpiWarps = 16;       // epilogue warps (4 per SM sub-partition)
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr uint64_t kTimeoutNs = 2000000000ull;   // 2 s per wait (drains: always)

struct TcArgs {
  int B, Hq, Hkv, G, w, P, rows, RC;  // RC: row chunks of 256
  int max_pages_per_seq, num_pages;
  const int32_t* block_table;
  const int32_t* slot_map;
  int64_t smax;                       // slot-map row length
  const int32_t* q_pos;
  const int32_t* attn_lo;
  const int32_t* attn_hi;
  const int32_t* out_lo;
  const int32_t* out_hi;
  int causal, accumulate, n_max;
  float* scores;
  int64_t scores_stride;
  float* part;      // [groups][RC*256][n_splits][2]
  float2* rowinfo;  // [groups][RC*256] {-lse2, qpos bits}
  int n_splits, tiles_per_split, tiles_per_cta2;
  int32_t* status;
  float scale;      // log2(e) / sqrt(D)
  const unsigned long long* limit;   // workspace bytes [0, 8): wait limit in ns, 0 = kTimeoutNs
  unsigned int* diag;                // workspace bytes [12, 16): first wait that gave up
};

// Limit of the producer's waits that give up (SE_ERR_TIMEOUT).  The MMA
// issuer's and the epilogue warps' waits keep kTimeoutNs (a runtime limit
// there measured 1-3 % slower) and end through the abort of the producer
// that feeds them; the drains (copies and MMAs in flight) always wait up to
// kTimeoutNs.
SE_DEV uint64_t wait_limit(const TcArgs& a) {
  const uint64_t v = a.limit != nullptr ? *a.limit : 0ull;
  return v != 0 ? v : kTimeoutNs;
}

// A producer wait: the limit is read only once a first try has failed.
SE_DEV bool producer_wait(uint64_t* bar, uint32_t parity, const TcArgs& a) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  return tc::mbar_wait(bar, parity, wait_limit(a));
}

// Key-tile geometry of one (sequence, group): tiles start at the page that
// holds attn_lo; tile t covers slots [base + 128 t, base + 128 t + 128).
struct TileGeom {
  int lo, hi, base, n_tiles, end_block;
  SE_DEV static TileGeom make(const TcArgs& a, int b) {
    TileGeom t;
    t.lo = a.attn_lo[b];
    t.hi = a.attn_hi[b];
    t.base = (t.lo / a.P) * a.P;
    t.n_tiles = t.hi > t.lo ? cdiv(t.hi - t.base, kKeyTile) : 0;
    t.end_block = cdiv(t.hi, a.P);
    return t;
  }
  SE_DEV int pages_in(int tile, int P) const {
    const int first = base / P + tile * (kKeyTile / P);
    return max(0, min(kKeyTile / P, end_block - first));
  }
};

SE_DEV bool geom_ok(const TcArgs& a, const TileGeom& t) {
  return t.lo >= 0 && t.hi >= t.lo && t.hi - t.lo <= a.n_max &&
         (int64_t)t.hi <= a.smax;
}

// Issues the TMA loads of K tile `tile` of (b, g) into `dst` (2 column halves
// of 128 rows x 128 bytes) and, when `pos` is set, the tile's key positions.
// Returns the bytes the loads will deliver.
SE_DEV uint32_t load_k_tile(const TcArgs& a, const CUtensorMap* kmap, const TileGeom& tg, int b,
                            int g, int tile, uint8_t* dst, int32_t* pos, uint64_t* bar) {
  const int P = a.P;
  const int np = tg.pages_in(tile, P);
  const int blk0 = tg.base / P + tile * (kKeyTile / P);
  uint32_t bytes = (uint32_t)np * P * kD * 2;
  if (pos != nullptr) {
    const int s0 = tg.base + tile * kKeyTile;
    const int cnt = (int)(a.smax - s0 < kKeyTile ? a.smax - s0 : kKeyTile);
    bytes += (uint32_t)cnt * 4;
  }
  tc::mbar_arrive_expect_tx(bar, bytes);
  const int32_t* bt = a.block_table + (int64_t)b * a.max_pages_per_seq;
  for (int i = 0; i < np; ++i) {
    const int page = bt[blk0 + i];
    const int y = (page * a.Hkv + g) * P;
    tc::tma_load_2d(dst + i * P * 128, kmap, bar, 0, y);
    tc::tma_load_2d(dst + kKTileBytes / 2 + i * P * 128, kmap, bar, 64, y);
  }
  if (pos != nullptr) {
    const int s0 = tg.base + tile * kKeyTile;
    const int cnt = (int)(a.smax - s0 < kKeyTile ? a.smax - s0 : kKeyTile);
    const int32_t* src = a.slot_map + ((int64_t)b * a.Hkv + g) * a.smax + s0;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(tc::smem_u32(pos)), "l"(src), "r"(cnt * 4), "r"(tc::smem_u32(bar))
        : "memory");
  }
  return bytes;
}

SE_DEV void load_q_chunk(const TcArgs& a, const CUtensorMap* qmap, int b, int g, int rc,
                         uint8_t* dst, uint64_t* bar) {
  const int qpc = kRowChunk / a.G;  // queries per chunk
  tc::mbar_arrive_expect_tx(bar, kQChunkBytes);
  tc::tma_load_4d(dst, qmap, bar, 0, g * a.G, rc * qpc, b);
  tc::tma_load_4d(dst + kQChunkBytes / 2, qmap, bar, 64, g * a.G, rc * qpc, b);
}

SE_DEV bool aborted(const int* flag) { return *reinterpret_cast<const volatile int*>(flag) != 0; }

SE_DEV void record_timeout(const TcArgs& a, int* s_abort) {
  set_status(a.status, SE_ERR_TIMEOUT);
  if (a.diag != nullptr)
    atomicCAS(a.diag, 0u, 1u + ((threadIdx.x >> 5) << 8 | (blockIdx.x & 0xffffu) << 16));
  atomicExch(s_abort, 1);
}

}  // namespace

constexpr int kMaxTilesPerSplit = 64;

// Largest query position of row chunk rc of sequence b (rows are (query, head)).
SE_DEV int chunk_max_qpos(const TcArgs& a, int b, int rc, int lane) {
  const int q0 = rc * (kRowChunk / a.G);
  const int q1 = min(q0 + kRowChunk / a.G, a.w);
  int mx = INT_MIN;
  for (int q = q0 + lane; q < q1; q += 32) mx = max(mx, a.q_pos[(int64_t)b * a.w + q]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  return mx;
}

// Smallest position among the keys of tile `tile` (slots in [lo, hi)).
SE_DEV int tile_min_pos(const TcArgs& a, const TileGeom& tg, int b, int g, int tile, int lane) {
  const int32_t* sm = a.slot_map + ((int64_t)b * a.Hkv + g) * a.smax;
  int mn = INT_MAX;
  for (int j = lane; j < kKeyTile; j += 32) {
    const int slot = tg.base + tile * kKeyTile + j;
    if (slot >= tg.lo && slot < tg.hi) mn = min(mn, sm[slot]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
  return mn;
}

// Fills list[0 .. *n) with the tiles of [t0, t0 + count) that at least one
// row of chunk rc can see (every tile when not causal).  Called by all
// threads of the CTA; the caller syncs before reading the list.
SE_DEV void active_tiles(const TcArgs& a, const TileGeom& tg, int b, int g, int rc, int t0,
                         int count, int* list, int* n) {
  __shared__ int s_keep[kMaxTilesPerSplit];
  __shared__ int s_qmax;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  count = min(count, kMaxTilesPerSplit);
  if (!a.causal) {
    if (threadIdx.x == 0) {
      for (int i = 0; i < count; ++i) list[i] = t0 + i;
      *n = count;
    }
    return;
  }
  if (warp == 0) {
    const int qm = chunk_max_qpos(a, b, rc, lane);
    if (lane == 0) s_qmax = qm;
  }
  __syncthreads();
  for (int i = warp; i < count; i += nw) {
    const int mn = tile_min_pos(a, tg, b, g, t0 + i, lane);
    if (lane == 0) s_keep[i] = mn <= s_qmax ? 1 : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int k = 0;
    for (int i = 0; i < count; ++i)
      if (s_keep[i]) list[k++] = t0 + i;
    *n = k;
  }
}

constexpr int kMaxRowChunkList = 1024;

// Fills list[0 .. *n) with the row chunks of [0, RC) in which some query can
// see some key of tiles [t0, t0 + count) (a chunk is dropped only when all its
// queries precede all those keys).  Returns false, leaving the list unused,
// when every chunk is kept anyway (not causal, or RC above the list size).
// Called by all threads of the CTA; the caller syncs before reading.
SE_DEV bool active_row_chunks(const TcArgs& a, const TileGeom& tg, int b, int g, int RC, int t0,
                              int count, int* list, int* n) {
  if (!a.causal || RC > kMaxRowChunkList) return false;
  __shared__ int s_kmin;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  if (threadIdx.x == 0) s_kmin = INT_MAX;
  __syncthreads();
  for (int i = warp; i < count; i += nw) {
    const int mn = tile_min_pos(a, tg, b, g, t0 + i, lane);
    if (lane == 0) atomicMin(&s_kmin, mn);
  }
  __syncthreads();
  for (int rc = warp; rc < RC; rc += nw) {
    const int qm = chunk_max_qpos(a, b, rc, lane);
    if (lane == 0) list[rc] = qm >= s_kmin ? 1 : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int k = 0;
    for (int rc = 0; rc < RC; ++rc)
      if (list[rc]) list[k++] = rc;
    *n = k;
  }
  return true;
}

// One block of N columns of a row for the online base-2 softmax statistics
// (m, l) of pass 1.  fast: every key of the block is in range and visible.
template <int N>
SE_DEV void rowstats_block(const uint32_t (&r)[N], bool fast, bool row_ok, int key0,
                           const TileGeom& tg, bool causal, const int32_t* pos, int qpos,
                           float scale, float& m, float& l) {
  if (fast) {
    float c0 = __uint_as_float(r[0]), c1 = __uint_as_float(r[1]);
#pragma unroll
    for (int j = 2; j < N; j += 4) {   // r[2..N-1] in pairs, two chains
      c0 = tc::fmax3(c0, __uint_as_float(r[j]), __uint_as_float(r[j + 1]));
      if (j + 2 < N) c1 = tc::fmax3(c1, __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
    }
    const float mn = fmaxf(m, fmaxf(c0, c1) * scale);
    const uint64_t sc2 = tc::f2(scale, scale), nm2 = tc::f2(-mn, -mn);
    uint64_t s01 = 0, s23 = 0;   // (+0, +0) pairs
#pragma unroll
    for (int j = 0; j < N; j += 4) {
      float a0, a1, b0, b1;
      tc::f2split(tc::ffma2(tc::f2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), sc2, nm2), a0, a1);
      tc::f2split(tc::ffma2(tc::f2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])), sc2, nm2), b0, b1);
      s01 = tc::fadd2(s01, tc::f2(tc::ex2(a0), tc::ex2(a1)));
      s23 = tc::fadd2(s23, tc::f2(tc::ex2(b0), tc::ex2(b1)));
    }
    float x0, x1, y0, y1;
    tc::f2split(s01, x0, x1);
    tc::f2split(s23, y0, y1);
    l = l * tc::ex2(m - mn) + ((x0 + x1) + (y0 + y1));
    m = mn;
    return;
  }
  float v[N];
  float c0 = -INFINITY, c1 = -INFINITY;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const int key = key0 + j;
    bool vis = row_ok && key >= tg.lo && key < tg.hi;
    if (causal) vis = vis && pos[j] <= qpos;
    v[j] = vis ? __uint_as_float(r[j]) * scale : -INFINITY;
    if (j & 1) c1 = fmaxf(c1, v[j]); else c0 = fmaxf(c0, v[j]);
  }
  const float cm = fmaxf(c0, c1);
  if (cm != -INFINITY) {
    const float mn = fmaxf(m, cm);
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int j = 0; j < N; j += 2) {
      s0 += tc::ex2(v[j] - mn);
      s1 += tc::ex2(v[j + 1] - mn);
    }
    l = l * tc::ex2(m - mn) + (s0 + s1);
    m = mn;
  }
}

// One 32-row block of a key's column sum in pass 2: adds
// exp2(logit * scale - lse2) over the rows that see the key (nlse holds
// -lse2 per row).  fast: every row of the chunk sees it.
template <int N>
SE_DEV void colsum_block(const uint32_t (&r)[N], bool fast, int kpos, const float* nlse,
                         const int* qp, float scale, float& cs0, float& cs1, float& cs2,
                         float& cs3) {
  if (fast) {
    const uint64_t sc2 = tc::f2(scale, scale);
    uint64_t s01 = tc::f2(cs0, cs1), s23 = tc::f2(cs2, cs3);
#pragma unroll
    for (int j = 0; j < N; j += 4) {
      const ulonglong2 nl = *reinterpret_cast<const ulonglong2*>(nlse + j);   // two pairs
      float a0, a1, b0, b1;
      tc::f2split(tc::ffma2(tc::f2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), sc2, nl.x),
                  a0, a1);
      tc::f2split(tc::ffma2(tc::f2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])), sc2, nl.y),
                  b0, b1);
      s01 = tc::fadd2(s01, tc::f2(tc::ex2(a0), tc::ex2(a1)));
      s23 = tc::fadd2(s23, tc::f2(tc::ex2(b0), tc::ex2(b1)));
    }
    tc::f2split(s01, cs0, cs1);
    tc::f2split(s23, cs2, cs3);
    return;
  }
#pragma unroll
  for (int j = 0; j < N; j += 2) {
    float p0 = tc::ex2(fmaf(__uint_as_float(r[j]), scale, nlse[j]));
    float p1 = tc::ex2(fmaf(__uint_as_float(r[j + 1]), scale, nlse[j + 1]));
    if (kpos > qp[j]) p0 = 0.f;
    if (kpos > qp[j + 1]) p1 = 0.f;
    cs0 += p0;
    cs1 += p1;
  }
}

// Column sum of one key over 32 NB rows held in TMEM at tb (lane = key,
// columns = rows), one 32-row block in registers at a time: the epilogue's
// sixteen warps cover the load latency (loading the next block while summing
// the current one measured slower).
template <int NB>
SE_DEV void colsum_tile_seq(uint32_t tb, bool fast, int kpos, const float* lse_s, const int* qp_s,
                            float scale, float& cs0, float& cs1, float& cs2, float& cs3) {
#pragma unroll 1
  for (int c = 0; c < NB; ++c) {
    uint32_t r[32];
    tc::tmem_ld32_async(tb + c * 32, r);
    tc::tmem_wait32(r);
    colsum_block(r, fast, kpos, lse_s + c * 32, qp_s + c * 32, scale, cs0, cs1, cs2, cs3);
  }
}

// ---------------------------------------------------------------------------
// Pass 1: row statistics.  grid (n_splits, RC, B*Hkv), 576 threads.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
score_rowstats_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                  TcArgs a) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_s = smem;                                   // 64 KB
  uint8_t* k_s = q_s + kQChunkBytes;                     // kStages1 x 32 KB
  int32_t* pos_s = reinterpret_cast<int32_t*>(k_s + kStages1 * kKTileBytes);  // [S][128]
  uint64_t* bars = reinterpret_cast<uint64_t*>(pos_s + kStages1 * kKeyTile);
  uint64_t* full = bars;                   // [S]  TMA -> MMA / epilogue
  uint64_t* empty = bars + kStages1;       // [S]  MMA done reading K
  uint64_t* pos_free = bars + 2 * kStages1;  // [S] epilogue done with positions
  uint64_t* acc_full = bars + 3 * kStages1;  // [2]
  uint64_t* acc_free = acc_full + 2;         // [2]
  uint64_t* q_full = acc_free + 2;
  uint64_t* done = q_full + 1;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x, rc = blockIdx.y, bg = blockIdx.z;
  const int b = bg / a.Hkv, g = bg % a.Hkv;
  const TileGeom tg = TileGeom::make(a, b);
  const bool ok = geom_ok(a, tg);
  const int t_begin = split * a.tiles_per_split;
  const int t_end = ok ? min(t_begin + a.tiles_per_split, tg.n_tiles) : 0;
  const int n_range = max(t_end - t_begin, 0);
  __shared__ int s_tiles[kMaxTilesPerSplit];   // tiles of the range that some row sees
  __shared__ int s_n;

  if (threadIdx.x == 0) {
    s_abort = 0;
    if (!ok) set_status(a.status, SE_ERR_BOUNDS);
    for (int s = 0; s < kStages1; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
      tc::mbar_init(&pos_free[s], kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_free[i], kEpiWarps);
    }
    tc::mbar_init(q_full, 1);
    tc::mbar_init(done, 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&s_tmem, 512);
  // causal: drop key tiles whose every key lies after the chunk's last query
  active_tiles(a, tg, b, g, rc, t_begin, n_range, s_tiles, &s_n);
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int n_my = s_n;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (tc::elect_one()) {
      tc::tma_prefetch_desc(&kmap);
      tc::tma_prefetch_desc(&qmap);
      if (n_my > 0) load_q_chunk(a, &qmap, b, g, rc, q_s, q_full);
      int issued = 0;
      for (int i = 0; i < n_my && !aborted(&s_abort); ++i) {
        const int s = i % kStages1;
        const uint32_t par = ((i / kStages1) & 1) ^ 1;
        if (i >= kStages1) {
          if (!producer_wait(&empty[s], par, a) ||
              !producer_wait(&pos_free[s], par, a)) {
            record_timeout(a, &s_abort);
            break;
          }
        }
        load_k_tile(a, &kmap, tg, b, g, s_tiles[i], k_s + s * kKTileBytes,
                    a.causal ? pos_s + s * kKeyTile : nullptr, &full[s]);
        issued = i + 1;
      }
      // drain: every issued load must land before the CTA can exit
      for (int i = max(0, issued - kStages1); i < issued; ++i)
        tc::mbar_wait(&full[i % kStages1], (i / kStages1) & 1, kTimeoutNs);
      if (n_my > 0) tc::mbar_wait(q_full, 0, kTimeoutNs);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (tc::elect_one()) {
      const uint32_t idesc = tc::idesc_bf16_f32(128, kKeyTile);
      bool go = n_my > 0 && tc::mbar_wait(q_full, 0, kTimeoutNs);
      if (n_my > 0 && !go) record_timeout(a, &s_abort);
      for (int i = 0; go && i < n_my && !aborted(&s_abort); ++i) {
        const int s = i % kStages1;
        const int acc = i & 1;
        if (!tc::mbar_wait(&full[s], (i / kStages1) & 1, kTimeoutNs) ||
            (i >= 2 && !tc::mbar_wait(&acc_free[acc], ((i >> 1) & 1) ^ 1, kTimeoutNs))) {
          record_timeout(a, &s_abort);
          break;
        }
        tc::tc_fence_after();
        const uint32_t kbase = tc::smem_u32(k_s + s * kKTileBytes);
        const uint32_t qbase = tc::smem_u32(q_s);
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t ad = tc::smem_desc_sw128(qbase + (k >> 2) * (kQChunkBytes / 2) +
                                                    mb * (128 * 128) + (k & 3) * 32);
            const uint64_t bd = tc::smem_desc_sw128(kbase + (k >> 2) * (kKTileBytes / 2) + (k & 3) * 32);
            tc::mma_bf16(tmem + acc * 256 + mb * 128, ad, bd, idesc, k > 0 ? 1u : 0u);
          }
        }
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&acc_full[acc]);
      }
      tc::mma_commit(done);
      tc::mbar_wait(done, 0, kTimeoutNs);
    }
  } else {
    // ---------------- epilogue: one row and column half per thread ----------------
    // 16 warps: (row block mb, TMEM lane quarter, column half of each tile)
    const int e = warp - 2;
    const int mb = (e >> 2) & 1;
    const int half = e >> 3;
    const int quarter = warp & 3;         // TMEM lane quarter this warp may read
    const int r = mb * 128 + quarter * 32 + lane;  // row in chunk
    const int row = rc * kRowChunk + r;
    const bool row_ok = row < a.rows;
    const int qpos = row_ok ? a.q_pos[(int64_t)b * a.w + row / a.G] : -1;
    float m = -INFINITY, l = 0.f;
    for (int i = 0; i < n_my; ++i) {
      const int s = i % kStages1;
      const int acc = i & 1;
      bool w_ok = tc::mbar_wait(&acc_full[acc], (i >> 1) & 1, kTimeoutNs);
      if (w_ok && a.causal) w_ok = tc::mbar_wait(&full[s], (i / kStages1) & 1, kTimeoutNs);
      // warp-uniform decision: tcgen05.ld below is a warp-collective
      if (!__all_sync(0xffffffffu, w_ok)) {
        record_timeout(a, &s_abort);
        break;
      }
      tc::tc_fence_after();
      const int tile = s_tiles[i];
      const int key0 = tg.base + tile * kKeyTile + half * 64;   // this warp's 64 columns
      const int32_t* pos = pos_s + s * kKeyTile + half * 64;
      // fast path: every key of the block is in range and visible to this row
      bool fast = row_ok && key0 >= tg.lo && key0 + 64 <= tg.hi;
      if (a.causal) {
        const int2 p2 = reinterpret_cast<const int2*>(pos)[lane];
        int mx = max(p2.x, p2.y);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        fast = fast && mx <= qpos;
      }
      {
        // two 32-column blocks; the second loads while the first is reduced
        uint32_t ra[32], rb[32];
        const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + acc * 256 + mb * 128 + half * 64;
        tc::tmem_ld32_async(tb, ra);
        tc::tmem_wait32(ra);
        tc::tmem_ld32_async(tb + 32, rb);
        rowstats_block(ra, fast, row_ok, key0, tg, a.causal, pos, qpos, a.scale, m, l);
        tc::tmem_wait32(rb);
        rowstats_block(rb, fast, row_ok, key0 + 32, tg, a.causal, pos + 32, qpos, a.scale, m, l);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&acc_free[acc]);
        tc::mbar_arrive(&pos_free[s]);
      }
    }
    if (row_ok) {
      float* p = a.part + (((int64_t)bg * a.RC * kRowChunk + row) * 2 * a.n_splits + 2 * split + half) * 2;
      p[0] = m;
      p[1] = l;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Row info: -lse2 per row (-inf when the row sees nothing) and query position.
// grid (cdiv(RC*256, 256), B*Hkv)
// ---------------------------------------------------------------------------
__global__ void score_rowinfo_tc(TcArgs a) {
  pdl_enter();
  const int bg = blockIdx.y, b = bg / a.Hkv;
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  const int padded = a.RC * kRowChunk;
  if (row >= padded) return;
  float lse = INFINITY;
  int qpos = 0x7fffffff;   // padded rows: lse = +inf already makes p = 0
  if (row < a.rows) {
    // two slots per split (the column halves of its tiles)
    const float* p = a.part + ((int64_t)bg * padded + row) * 2 * a.n_splits * 2;
    float M = -INFINITY;
    for (int s = 0; s < 2 * a.n_splits; ++s) M = fmaxf(M, p[2 * s]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int s = 0; s < 2 * a.n_splits; ++s) L += p[2 * s + 1] * exp2f(p[2 * s] - M);
    if (L > 0.f) lse = M + log2f(L);
    qpos = a.q_pos[(int64_t)b * a.w + row / a.G];
  }
  // per 256-row chunk: 256 lse2 values, then 256 query positions
  float* chunk = reinterpret_cast<float*>(a.rowinfo + (int64_t)bg * padded + (row / kRowChunk) * kRowChunk);
  chunk[row % kRowChunk] = -lse;   // stored negated: the FMA adds it
  chunk[kRowChunk + row % kRowChunk] = __int_as_float(qpos);
}

// ---------------------------------------------------------------------------
// Pass 2: column sums.  grid (cdiv(n_tiles_max, tiles_per_cta2), B*Hkv).
// Key tiles are taken in pairs (2p, 2p+1); for each row chunk rc the pair is
// multiplied by the same Q chunk, tile 2p into TMEM buffer 0 and tile 2p+1
// into buffer 1.  Half the epilogue warps own even tiles, half odd tiles; a
// thread sums one key over its row half of every chunk in registers.  When the rows
// fit one chunk the Q chunk stays resident and K tiles stream through four
// stages; otherwise Q chunks stream through two stages (once per pair) and K
// uses two stages.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
score_colsum_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                TcArgs a) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int RC = a.RC;
  const bool q_resident = RC == 1;
  const int QS = q_resident ? 1 : 2;       // Q stages
  const int KS = q_resident ? 4 : 2;       // K stages
  uint8_t* q_s = smem;
  uint8_t* k_s = q_s + QS * kQChunkBytes;
  int32_t* pos_s = reinterpret_cast<int32_t*>(k_s + KS * kKTileBytes);   // [KS][128]
  float2* info_s = reinterpret_cast<float2*>(pos_s + KS * kKeyTile);     // [QS][256]
  uint64_t* bars = reinterpret_cast<uint64_t*>(info_s + QS * kRowChunk);
  uint64_t* kfull = bars;                 // [KS]
  uint64_t* kempty = bars + 4;            // [KS] MMA done with the K tile
  uint64_t* pfree = bars + 8;             // [KS] epilogue done with its positions
  uint64_t* qfull = bars + 12;            // [QS]
  uint64_t* qempty = bars + 14;           // [QS] MMA done with the Q chunk
  uint64_t* ifree = bars + 16;            // [QS] epilogue done with the row info
  uint64_t* acc_full = bars + 18;         // [2]
  uint64_t* acc_free = bars + 20;         // [2]
  uint64_t* done = bars + 22;
  uint64_t* hfull = bars + 23;            // [set][buf] the second row half's sums are in s_half
  uint64_t* hempty = bars + 27;           // [set][buf] the first row half has read them
  __shared__ float s_half[2][2][kKeyTile];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bg = blockIdx.y, b = bg / a.Hkv, g = bg % a.Hkv;
  const TileGeom tg = TileGeom::make(a, b);
  const bool ok = geom_ok(a, tg);
  const int t_begin = blockIdx.x * a.tiles_per_cta2;
  const int t_end = ok ? min(t_begin + a.tiles_per_cta2, tg.n_tiles) : 0;
  const int n_my = max(t_end - t_begin, 0);
  const int n_pairs = cdiv(n_my, 2);
  __shared__ int s_rcs[kMaxRowChunkList];   // row chunks that see some key of this CTA
  __shared__ int s_nrc;

  if (threadIdx.x == 0) {
    s_abort = 0;
    if (!ok) set_status(a.status, SE_ERR_BOUNDS);
    for (int s = 0; s < KS; ++s) {
      tc::mbar_init(&kfull[s], 1);
      tc::mbar_init(&kempty[s], 1);
      tc::mbar_init(&pfree[s], kEpiWarps / 2);
    }
    for (int i = 0; i < QS; ++i) {
      tc::mbar_init(&qfull[i], 1);
      tc::mbar_init(&qempty[i], 1);
      tc::mbar_init(&ifree[i], kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_free[i], kEpiWarps / 2);
    }
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(&hfull[i], 4);
      tc::mbar_init(&hempty[i], 4);
    }
    tc::mbar_init(done, 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&s_tmem, 512);
  // causal: drop row chunks whose every query precedes every key of this CTA
  const bool rc_list = active_row_chunks(a, tg, b, g, RC, t_begin, n_my, s_rcs, &s_nrc);
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int n_rc = rc_list ? s_nrc : RC;
  const float2* info_g = a.rowinfo + (int64_t)bg * RC * kRowChunk;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (tc::elect_one()) {
      tc::tma_prefetch_desc(&kmap);
      tc::tma_prefetch_desc(&qmap);
      int k_issued = 0, q_issued = 0;
      bool stop = false;
      for (int p = 0; p < n_pairs && !stop && !aborted(&s_abort); ++p) {
        for (int ri = 0; ri < n_rc && !stop; ++ri) {
          const int rc = rc_list ? s_rcs[ri] : ri;
          if (ri == 0) {
            for (int t = 2 * p; t < min(2 * p + 2, n_my); ++t) {
              const int s = t % KS;
              const uint32_t par = ((t / KS) & 1) ^ 1;
              if (t >= KS && (!producer_wait(&kempty[s], par, a) ||
                              !producer_wait(&pfree[s], par, a))) {
                record_timeout(a, &s_abort);
                stop = true;
                break;
              }
              load_k_tile(a, &kmap, tg, b, g, t_begin + t, k_s + s * kKTileBytes,
                          a.causal ? pos_s + s * kKeyTile : nullptr, &kfull[s]);
              k_issued = t + 1;
            }
            if (stop) break;
          }
          if (q_resident && q_issued > 0) continue;
          const int qs = q_issued % QS;
          const uint32_t par = ((q_issued / QS) & 1) ^ 1;
          if (q_issued >= QS && (!producer_wait(&qempty[qs], par, a) ||
                                 !producer_wait(&ifree[qs], par, a))) {
            record_timeout(a, &s_abort);
            stop = true;
            break;
          }
          tc::mbar_arrive_expect_tx(&qfull[qs], kQChunkBytes + kRowChunk * 8);
          const int qpc = kRowChunk / a.G;
          tc::tma_load_4d(q_s + qs * kQChunkBytes, &qmap, &qfull[qs], 0, g * a.G, rc * qpc, b);
          tc::tma_load_4d(q_s + qs * kQChunkBytes + kQChunkBytes / 2, &qmap, &qfull[qs], 64,
                          g * a.G, rc * qpc, b);
          asm volatile(
              "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
              ::"r"(tc::smem_u32(info_s + qs * kRowChunk)), "l"(info_g + rc * kRowChunk),
              "r"(kRowChunk * 8), "r"(tc::smem_u32(&qfull[qs]))
              : "memory");
          q_issued++;
        }
      }
      for (int t = max(0, k_issued - KS); t < k_issued; ++t)
        tc::mbar_wait(&kfull[t % KS], (t / KS) & 1, kTimeoutNs);
      for (int j = max(0, q_issued - QS); j < q_issued; ++j)
        tc::mbar_wait(&qfull[j % QS], (j / QS) & 1, kTimeoutNs);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (tc::elect_one()) {
      const uint32_t idesc = tc::idesc_bf16_f32(128, kRowChunk);
      int q_used = 0;
      int uses[2] = {0, 0};
      bool stop = false;
      for (int p = 0; p < n_pairs && !stop && !aborted(&s_abort); ++p) {
        for (int ri = 0; ri < n_rc && !stop; ++ri) {
          const int qs = q_used % QS;
          if (!q_resident || q_used == 0) {
            if (!(q_resident && q_used > 0) &&
                !tc::mbar_wait(&qfull[qs], (q_used / QS) & 1, kTimeoutNs)) {
              record_timeout(a, &s_abort);
              stop = true;
              break;
            }
          }
          const int t1 = min(2 * p + 2, n_my);
          for (int t = 2 * p; t < t1; ++t) {
            const int s = t % KS;
            const int buf = t & 1;
            bool w_ok = true;
            if (ri == 0) w_ok = tc::mbar_wait(&kfull[s], (t / KS) & 1, kTimeoutNs);
            if (w_ok && uses[buf] > 0)
              w_ok = tc::mbar_wait(&acc_free[buf], (uses[buf] - 1) & 1, kTimeoutNs);
            if (!w_ok) {
              record_timeout(a, &s_abort);
              stop = true;
              break;
            }
            tc::tc_fence_after();
            const uint32_t kbase = tc::smem_u32(k_s + s * kKTileBytes);
            const uint32_t qbase = tc::smem_u32(q_s + qs * kQChunkBytes);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t ad = tc::smem_desc_sw128(kbase + (k >> 2) * (kKTileBytes / 2) + (k & 3) * 32);
              const uint64_t bd = tc::smem_desc_sw128(qbase + (k >> 2) * (kQChunkBytes / 2) + (k & 3) * 32);
              tc::mma_bf16(tmem + buf * 256, ad, bd, idesc, k > 0 ? 1u : 0u);
            }
            if (ri == n_rc - 1) tc::mma_commit(&kempty[s]);
            tc::mma_commit(&acc_full[buf]);
            uses[buf]++;
          }
          if (stop) break;
          if (!q_resident) tc::mma_commit(&qempty[qs]);
          q_used++;
        }
      }
      tc::mma_commit(done);
      tc::mbar_wait(done, 0, kTimeoutNs);
    }
  } else {
    // ---------------- epilogue: one key and row half per thread ----------------
    // 16 warps: (tile parity set: 0 even tiles / TMEM buffer 0, 1 odd tiles;
    // TMEM lane quarter; row half of each chunk).  The second half hands its
    // column sums to the first through s_half at the end of each pair.
    const int e = warp - 2;
    const int set = (e >> 2) & 1;
    const int half = e >> 3;
    const int quarter = warp & 3;
    const int kl = quarter * 32 + lane;   // key within its tile
    int use = 0;
    bool stop = false;
    for (int p = 0; p < n_pairs && !stop; ++p) {
      const int t = 2 * p + set;
      const int s = t % KS;
      if (t >= n_my) {
        // no tile of this parity in the last pair: still release each streamed
        // Q chunk after it has landed, so the pair's row-info stage frees up
        if (!q_resident) {
          for (int ri = 0; ri < n_rc; ++ri) {
            const int qn = p * n_rc + ri;
            if (!__all_sync(0xffffffffu, tc::mbar_wait(&qfull[qn % QS], (qn / QS) & 1, kTimeoutNs))) {
              record_timeout(a, &s_abort);
              stop = true;
              break;
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&ifree[qn % QS]);
          }
        }
        break;
      }
      float colsum = 0.f;
      int kpos = 0;
      for (int ri = 0; ri < n_rc; ++ri) {
        const int qn = p * n_rc + ri;        // Q chunk load number (0 when resident)
        const int qs = q_resident ? 0 : qn % QS;
        bool w_ok = tc::mbar_wait(&acc_full[set], use & 1, kTimeoutNs);
        if (w_ok && ri == 0 && a.causal) w_ok = tc::mbar_wait(&kfull[s], (t / KS) & 1, kTimeoutNs);
        if (w_ok) w_ok = tc::mbar_wait(&qfull[qs], q_resident ? 0 : ((qn / QS) & 1), kTimeoutNs);
        if (!__all_sync(0xffffffffu, w_ok)) {  // tcgen05.ld below is a warp-collective
          record_timeout(a, &s_abort);
          stop = true;
          break;
        }
        tc::tc_fence_after();
        if (ri == 0 && a.causal) kpos = pos_s[s * kKeyTile + kl];
        const float* lse_s = reinterpret_cast<const float*>(info_s + qs * kRowChunk) + half * 128;
        const int* qp_s = reinterpret_cast<const int*>(info_s + qs * kRowChunk) + kRowChunk + half * 128;
        // fast path: this key is visible to every row of the half chunk
        bool fast = !a.causal;
        if (a.causal) {
          const int4 q4 = reinterpret_cast<const int4*>(qp_s)[lane];
          int mn = min(min(q4.x, q4.y), min(q4.z, q4.w));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
          fast = kpos <= mn;
        }
        float cs0 = 0.f, cs1 = 0.f, cs2 = 0.f, cs3 = 0.f;
        colsum_tile_seq<4>(tmem + ((uint32_t)(quarter * 32) << 16) + set * 256 + half * 128, fast,
                           kpos, lse_s, qp_s, a.scale, cs0, cs1, cs2, cs3);
        colsum += (cs0 + cs1) + (cs2 + cs3);
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&acc_free[set]);
          if (!q_resident) tc::mbar_arrive(&ifree[qs]);
          if (ri == n_rc - 1) tc::mbar_arrive(&pfree[s]);
        }
        use++;
      }
      if (stop) break;
      // the two row halves meet: buffer p & 1 of this set, its (p >> 1)-th use
      const int hb = set * 2 + (p & 1), k_use = p >> 1;
      if (half == 1) {
        const bool ok_e = k_use == 0 || tc::mbar_wait(&hempty[hb], (k_use - 1) & 1, kTimeoutNs);
        if (!__all_sync(0xffffffffu, ok_e)) {
          record_timeout(a, &s_abort);
          break;
        }
        s_half[set][p & 1][kl] = colsum;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&hfull[hb]);
        continue;
      }
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&hfull[hb], k_use & 1, kTimeoutNs))) {
        record_timeout(a, &s_abort);
        break;
      }
      colsum += s_half[set][p & 1][kl];
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&hempty[hb]);
      const int key = tg.base + (t_begin + t) * kKeyTile + kl;
      if (key >= a.out_lo[b] && key < a.out_hi[b] && key >= tg.lo && key < tg.hi &&
          key < a.scores_stride) {
        float* out = a.scores + (int64_t)bg * a.scores_stride + key;
        *out = a.accumulate ? *out + colsum : colsum;
      }
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}


SE_DEV int group_tiles(const TcArgs& a, int bg) {
  const TileGeom tg = TileGeom::make(a, bg / a.Hkv);
  return geom_ok(a, tg) ? tg.n_tiles : 0;
}


// ---------------------------------------------------------------------------
// Pass 1, persistent form for one row chunk (RC == 1).  grid = the number of
// SMs; CTA c takes an equal share of the global (group, tile) sequence, a
// group change counted as kSwitchTiles tiles (cta_tiles).  Each epilogue thread keeps its row's running max / sum per group
// and writes it, when the group ends in this CTA, to the partial slots of
// this CTA: part[(group * 256 + row) * 2C + 2c + half].  The persistent pass 2
// merges the slots of the CTAs whose ranges meet a group when it starts it.
// ---------------------------------------------------------------------------
constexpr int kMaxGroupsP = 2048;   // groups the persistent passes index in shared memory

// s_pre[x] = key tiles of groups 0 .. x-1, s_pre[groups] = all tiles.  Called
// by every thread of the CTA (it synchronises the CTA).
SE_DEV void group_prefix(const TcArgs& a, int* s_pre) {
  const int groups = a.B * a.Hkv;
  for (int x = threadIdx.x; x < groups; x += blockDim.x) s_pre[x + 1] = group_tiles(a, x);
  if (threadIdx.x == 0) s_pre[0] = 0;
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int carry = 0;
    for (int base = 0; base < groups; base += 32) {
      const int i = base + lane;
      int v = i < groups ? s_pre[i + 1] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
      }
      if (i < groups) s_pre[i + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
}

// Group holding global tile x (x < s_pre[groups]) and the tile within it.
SE_DEV void locate_pre(const int* s_pre, int groups, int x, int& bg, int& tile) {
  int lo = 0, hi = groups;            // largest g with s_pre[g] <= x
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (s_pre[mid] <= x) lo = mid; else hi = mid;
  }
  bg = lo;
  while (bg < groups - 1 && s_pre[bg + 1] <= x) ++bg;   // skip empty groups
  tile = x - s_pre[bg];
}

// The CTA whose range [c T / C, (c+1) T / C) holds work coordinate x.
SE_DEV int cta_of(int64_t x, int64_t T, int64_t C) { return (int)(((x + 1) * C - 1) / T); }

// The persistent passes split work coordinates, not tiles, evenly over the
// CTAs: tile t of group g sits at t + kSwitchTiles * g, so a CTA whose range
// crosses into a new group takes kSwitchTiles fewer tiles.  The change costs
// the CTA a Q load, a pipeline drain and refill and, in pass 2, the merge of
// the group's row statistics: on the SnapKV shape (32 groups of 256 tiles
// over 152 CTAs) 2 measured no gain, 4 and 6 cut the two passes by 4 and
// 6 us, 8 no further.
constexpr int kSwitchTiles = 6;

SE_DEV int64_t work_total(const int* s_pre, int groups) {
  return s_pre[groups] + (int64_t)kSwitchTiles * groups;
}

// Work coordinate of global tile x of group bg.
SE_DEV int64_t work_of(int x, int bg) { return x + (int64_t)kSwitchTiles * bg; }

// The first global tile whose work coordinate is at least X (all tiles, if
// none): the first group whose last tile reaches X, from there.
SE_DEV int tile_at_work(const int* s_pre, int groups, int64_t X) {
  int lo = 0, hi = groups;   // smallest bg with work_of(last tile of bg) >= X, groups if none
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (work_of(s_pre[mid + 1] - 1, mid) >= X) hi = mid; else lo = mid + 1;
  }
  if (lo == groups) return s_pre[groups];
  return (int)max((int64_t)s_pre[lo], X - (int64_t)kSwitchTiles * lo);
}

// The CTA's tile range [x0, x1) of the global (group, tile) sequence.
SE_DEV void cta_tiles(const int* s_pre, int groups, int& x0, int& x1) {
  const int64_t TW = work_total(s_pre, groups);
  x0 = tile_at_work(s_pre, groups, (int64_t)blockIdx.x * TW / gridDim.x);
  x1 = tile_at_work(s_pre, groups, (int64_t)(blockIdx.x + 1) * TW / gridDim.x);
}

__global__ void __launch_bounds__(kThreads, 1)
score_rowstats_persistent_tc(const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap qmap, TcArgs a) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int KS = kStages1;
  uint8_t* q_s = smem;
  uint8_t* k_s = q_s + kQChunkBytes;
  int32_t* pos_s = reinterpret_cast<int32_t*>(k_s + KS * kKTileBytes);
  uint64_t* bars = reinterpret_cast<uint64_t*>(pos_s + KS * kKeyTile);
  uint64_t* full = bars;             // [KS]
  uint64_t* empty = bars + 4;        // [KS]
  uint64_t* pos_free = bars + 8;     // [KS]
  uint64_t* acc_full = bars + 12;    // [2]
  uint64_t* acc_free = bars + 14;    // [2]
  uint64_t* q_full = bars + 16;
  uint64_t* q_done = bars + 17;
  uint64_t* done = bars + 18;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_range[2];

  __shared__ int s_pre[kMaxGroupsP + 1];
  const int groups = a.B * a.Hkv;
  group_prefix(a, s_pre);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_abort = 0;
    cta_tiles(s_pre, groups, s_range[0], s_range[1]);
    for (int i = 0; i < KS; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 1);
      tc::mbar_init(&pos_free[i], kEpiWarps);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_free[i], kEpiWarps);
    }
    tc::mbar_init(q_full, 1);
    tc::mbar_init(q_done, 1);
    tc::mbar_init(done, 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&s_tmem, 512);
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int x0 = s_range[0], x1 = s_range[1];
  const int n_my = x1 - x0;

  if (warp == 0) {
    if (tc::elect_one()) {
      tc::tma_prefetch_desc(&kmap);
      tc::tma_prefetch_desc(&qmap);
      int bg = 0, tile = 0;
      if (n_my > 0) locate_pre(s_pre, groups, x0, bg, tile);
      int cur = -1, gi = 0, issued = 0;
      for (int i = 0; i < n_my && !aborted(&s_abort); ++i) {
        while (tile >= s_pre[bg + 1] - s_pre[bg]) { ++bg; tile = 0; }
        const int b = bg / a.Hkv, g = bg % a.Hkv;
        if (bg != cur) {
          if (gi > 0 && !producer_wait(q_done, (gi - 1) & 1, a)) {
            record_timeout(a, &s_abort);
            break;
          }
          load_q_chunk(a, &qmap, b, g, 0, q_s, q_full);
          cur = bg;
          ++gi;
        }
        const int s = i % KS;
        const uint32_t par = ((i / KS) & 1) ^ 1;
        if (i >= KS && (!producer_wait(&empty[s], par, a) ||
                        !producer_wait(&pos_free[s], par, a))) {
          record_timeout(a, &s_abort);
          break;
        }
        const TileGeom tg = TileGeom::make(a, b);
        load_k_tile(a, &kmap, tg, b, g, tile, k_s + s * kKTileBytes,
                    a.causal ? pos_s + s * kKeyTile : nullptr, &full[s]);
        issued = i + 1;
        ++tile;
      }
      for (int i = max(0, issued - KS); i < issued; ++i)
        tc::mbar_wait(&full[i % KS], (i / KS) & 1, kTimeoutNs);
      if (gi > 0) tc::mbar_wait(q_full, (gi - 1) & 1, kTimeoutNs);
    }
  } else if (warp == 1) {
    if (tc::elect_one()) {
      const uint32_t idesc = tc::idesc_bf16_f32(128, kKeyTile);
      int bg = 0, tile = 0;
      if (n_my > 0) locate_pre(s_pre, groups, x0, bg, tile);
      int cur = -1, gi = 0;
      for (int i = 0; i < n_my && !aborted(&s_abort); ++i) {
        while (tile >= s_pre[bg + 1] - s_pre[bg]) { ++bg; tile = 0; }
        if (bg != cur) {
          if (gi > 0) tc::mma_commit(q_done);
          if (!tc::mbar_wait(q_full, gi & 1, kTimeoutNs)) {
            record_timeout(a, &s_abort);
            break;
          }
          cur = bg;
          ++gi;
        }
        const int s = i % KS;
        const int acc = i & 1;
        if (!tc::mbar_wait(&full[s], (i / KS) & 1, kTimeoutNs) ||
            (i >= 2 && !tc::mbar_wait(&acc_free[acc], ((i >> 1) & 1) ^ 1, kTimeoutNs))) {
          record_timeout(a, &s_abort);
          break;
        }
        tc::tc_fence_after();
        const uint32_t kbase = tc::smem_u32(k_s + s * kKTileBytes);
        const uint32_t qbase = tc::smem_u32(q_s);
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t ad = tc::smem_desc_sw128(qbase + (k >> 2) * (kQChunkBytes / 2) +
                                                    mb * (128 * 128) + (k & 3) * 32);
            const uint64_t bd = tc::smem_desc_sw128(kbase + (k >> 2) * (kKTileBytes / 2) + (k & 3) * 32);
            tc::mma_bf16(tmem + acc * 256 + mb * 128, ad, bd, idesc, k > 0 ? 1u : 0u);
          }
        }
        tc::mma_commit(&empty[s]);
        tc::mma_commit(&acc_full[acc]);
        ++tile;
      }
      tc::mma_commit(done);
      tc::mbar_wait(done, 0, kTimeoutNs);
    }
  } else {
    // 16 warps: (row block mb, TMEM lane quarter, column half of each tile)
    const int e = warp - 2;
    const int mb = (e >> 2) & 1;
    const int half = e >> 3;
    const int quarter = warp & 3;
    const int r = mb * 128 + quarter * 32 + lane;   // row of the group
    const bool row_ok = r < a.rows;
    int bg = 0, tile = 0;
    if (n_my > 0) locate_pre(s_pre, groups, x0, bg, tile);
    int cur = -1, qpos = -1;
    float m = -INFINITY, l = 0.f;
    for (int i = 0; i < n_my; ++i) {
      while (tile >= s_pre[bg + 1] - s_pre[bg]) { ++bg; tile = 0; }
      const int b = bg / a.Hkv;
      if (bg != cur) {
        if (cur >= 0 && row_ok) {
          float* p = a.part + (((int64_t)cur * kRowChunk + r) * 2 * gridDim.x + 2 * blockIdx.x + half) * 2;
          p[0] = m;
          p[1] = l;
        }
        m = -INFINITY;
        l = 0.f;
        qpos = row_ok ? a.q_pos[(int64_t)b * a.w + r / a.G] : -1;
        cur = bg;
      }
      const int s = i % KS;
      const int acc = i & 1;
      bool w_ok = tc::mbar_wait(&acc_full[acc], (i >> 1) & 1, kTimeoutNs);
      if (w_ok && a.causal) w_ok = tc::mbar_wait(&full[s], (i / KS) & 1, kTimeoutNs);
      if (!__all_sync(0xffffffffu, w_ok)) {
        record_timeout(a, &s_abort);
        break;
      }
      tc::tc_fence_after();
      const TileGeom tg = TileGeom::make(a, b);
      const int key0 = tg.base + tile * kKeyTile + half * 64;   // this warp's 64 columns
      const int32_t* pos = pos_s + s * kKeyTile + half * 64;
      bool fast = row_ok && key0 >= tg.lo && key0 + 64 <= tg.hi;
      if (a.causal) {
        const int2 p2 = reinterpret_cast<const int2*>(pos)[lane];
        int mx = max(p2.x, p2.y);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        fast = fast && mx <= qpos;
      }
      {
        // two 32-column blocks; the second loads while the first is reduced
        uint32_t ra[32], rb[32];
        const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + acc * 256 + mb * 128 + half * 64;
        tc::tmem_ld32_async(tb, ra);
        tc::tmem_wait32(ra);
        tc::tmem_ld32_async(tb + 32, rb);
        rowstats_block(ra, fast, row_ok, key0, tg, a.causal, pos, qpos, a.scale, m, l);
        tc::tmem_wait32(rb);
        rowstats_block(rb, fast, row_ok, key0 + 32, tg, a.causal, pos + 32, qpos, a.scale, m, l);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&acc_free[acc]);
        tc::mbar_arrive(&pos_free[s]);
      }
      ++tile;
    }
    if (cur >= 0 && row_ok) {
      float* p = a.part + (((int64_t)cur * kRowChunk + r) * 2 * gridDim.x + 2 * blockIdx.x + half) * 2;
      p[0] = m;
      p[1] = l;
    }
    // fewer tiles than CTAs: a CTA with an empty range may sit inside the
    // span of the group that holds the next tile, and pass 2 merges the slots
    // of every CTA in that span, so its slots of that group read as empty
    if (n_my == 0 && x0 < s_pre[groups] && row_ok) {
      int bg0 = 0, t0 = 0;
      locate_pre(s_pre, groups, x0, bg0, t0);
      float* p = a.part + (((int64_t)bg0 * kRowChunk + r) * 2 * gridDim.x + 2 * blockIdx.x + half) * 2;
      p[0] = -INFINITY;
      p[1] = 0.f;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}


// lse2 of row r of group bg from pass 1's partial slots (two per CTA whose
// tile range meets the group; n_ctas CTAs ran pass 1); +inf when the row saw
// no key.
SE_DEV float row_lse2(const TcArgs& a, const int* s_pre, int groups, int bg, int r, int n_ctas) {
  const int64_t TW = work_total(s_pre, groups);
  const int gstart = s_pre[bg];
  const int n = s_pre[bg + 1] - s_pre[bg];
  if (n <= 0 || s_pre[groups] <= 0) return INFINITY;
  const int first = cta_of(work_of(gstart, bg), TW, n_ctas);
  const int last = cta_of(work_of(gstart + n - 1, bg), TW, n_ctas);
  const float* p = a.part + ((int64_t)bg * kRowChunk + r) * 2 * n_ctas * 2;
  float M = -INFINITY;
  for (int c = 2 * first; c <= 2 * last + 1; ++c) M = fmaxf(M, p[2 * c]);
  float L = 0.f;
  if (M != -INFINITY)
    for (int c = 2 * first; c <= 2 * last + 1; ++c) L += p[2 * c + 1] * exp2f(p[2 * c] - M);
  return L > 0.f ? M + log2f(L) : INFINITY;
}

// ---------------------------------------------------------------------------
// Pass 2, persistent form for one row chunk (RC == 1: w * G <= 256 rows).
// grid = the number of SMs; CTA c takes the contiguous share of the global
// sequence of (group, key tile) pairs that pass 1 took (cta_tiles), so the
// last wave is full and the pipeline runs across tiles of consecutive groups
// without refilling.  The Q
// chunk and row info of a group are loaded when the group changes (after the
// MMA and both epilogue sets are done with the previous ones).  One set of
// eight epilogue warps takes the CTA's even local tiles (TMEM buffer 0), the
// other the odd ones; within a set, the two row halves of a key meet in
// shared memory.  Each CTA walks its tile range backwards: pass 1 walked it
// forwards, so the first tiles pass 2 needs are the ones pass 1 loaded last,
// the most likely to be still in L2.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
score_colsum_persistent_tc(const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap qmap, TcArgs a) {
  // Of pass 1's output this kernel reads only the partial row statistics, in
  // the epilogue warps; everything else it reads was written before pass 1
  // started (pass 1 began with its own wait for those writers).  So only the
  // epilogue waits for pass 1: the set-up, the Q and K loads and the first
  // MMAs overlap pass 1's last CTAs.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int KS = 4;
  uint8_t* q_s = smem;
  uint8_t* k_s = q_s + kQChunkBytes;
  int32_t* pos_s = reinterpret_cast<int32_t*>(k_s + KS * kKTileBytes);   // [KS][128]
  float2* info_s = reinterpret_cast<float2*>(pos_s + KS * kKeyTile);     // [256]
  uint64_t* bars = reinterpret_cast<uint64_t*>(info_s + kRowChunk);
  uint64_t* kfull = bars;            // [KS]
  uint64_t* kempty = bars + 4;       // [KS]
  uint64_t* pfree = bars + 8;        // [KS]
  uint64_t* qfull = bars + 12;
  uint64_t* qdone = bars + 13;       // MMA done with the group's Q
  uint64_t* ifree = bars + 14;       // every epilogue warp done with the group's row info
  uint64_t* acc_full = bars + 15;    // [2]
  uint64_t* acc_free = bars + 17;    // [2]
  uint64_t* done = bars + 19;
  uint64_t* hfull = bars + 20;       // [set][buf] the second row half's sums are in s_half
  uint64_t* hempty = bars + 24;      // [set][buf] the first row half has read them
  uint64_t* ifull = bars + 28;       // the group's row info is in info_s
  __shared__ float s_half[2][2][kKeyTile];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_range[2];

  __shared__ int s_pre[kMaxGroupsP + 1];
  const int groups = a.B * a.Hkv;
  group_prefix(a, s_pre);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    s_abort = 0;
    cta_tiles(s_pre, groups, s_range[0], s_range[1]);
    for (int i = 0; i < KS; ++i) {
      tc::mbar_init(&kfull[i], 1);
      tc::mbar_init(&kempty[i], 1);
      tc::mbar_init(&pfree[i], kEpiWarps / 2);
    }
    tc::mbar_init(qfull, 1);
    tc::mbar_init(qdone, 1);
    tc::mbar_init(ifree, kEpiWarps);
    tc::mbar_init(ifull, kRowChunk / 32);
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&acc_full[i], 1);
      tc::mbar_init(&acc_free[i], kEpiWarps / 2);
    }
    for (int i = 0; i < 4; ++i) {
      tc::mbar_init(&hfull[i], 4);
      tc::mbar_init(&hempty[i], 4);
    }
    tc::mbar_init(done, 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&s_tmem, 512);
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int x0 = s_range[0], x1 = s_range[1];
  const int n_my = x1 - x0;

  if (warp == 0) {
    // ---------------- producer ----------------
    if (tc::elect_one()) {
      tc::tma_prefetch_desc(&kmap);
      tc::tma_prefetch_desc(&qmap);
      int bg = 0, tile = 0;
      if (n_my > 0) locate_pre(s_pre, groups, x1 - 1, bg, tile);
      int cur = -1, gi = 0, issued = 0;
      for (int lt = 0; lt < n_my && !aborted(&s_abort); ++lt) {
        while (tile < 0) { --bg; tile = s_pre[bg + 1] - s_pre[bg] - 1; }
        const int b = bg / a.Hkv, g = bg % a.Hkv;
        if (bg != cur) {
          if (gi > 0 && !producer_wait(qdone, (gi - 1) & 1, a)) {
            record_timeout(a, &s_abort);
            break;
          }
          tc::mbar_arrive_expect_tx(qfull, kQChunkBytes);
          tc::tma_load_4d(q_s, &qmap, qfull, 0, g * a.G, 0, b);
          tc::tma_load_4d(q_s + kQChunkBytes / 2, &qmap, qfull, 64, g * a.G, 0, b);
          cur = bg;
          ++gi;
        }
        const int s = lt % KS;
        const uint32_t par = ((lt / KS) & 1) ^ 1;
        if (lt >= KS && (!producer_wait(&kempty[s], par, a) ||
                         !producer_wait(&pfree[s], par, a))) {
          record_timeout(a, &s_abort);
          break;
        }
        const TileGeom tg = TileGeom::make(a, b);
        load_k_tile(a, &kmap, tg, b, g, tile, k_s + s * kKTileBytes,
                    a.causal ? pos_s + s * kKeyTile : nullptr, &kfull[s]);
        issued = lt + 1;
        --tile;
      }
      for (int i = max(0, issued - KS); i < issued; ++i)
        tc::mbar_wait(&kfull[i % KS], (i / KS) & 1, kTimeoutNs);
      if (gi > 0) tc::mbar_wait(qfull, (gi - 1) & 1, kTimeoutNs);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (tc::elect_one()) {
      const uint32_t idesc = tc::idesc_bf16_f32(128, kRowChunk);
      int bg = 0, tile = 0;
      if (n_my > 0) locate_pre(s_pre, groups, x1 - 1, bg, tile);
      int cur = -1, gi = 0;
      int uses[2] = {0, 0};
      for (int lt = 0; lt < n_my && !aborted(&s_abort); ++lt) {
        while (tile < 0) { --bg; tile = s_pre[bg + 1] - s_pre[bg] - 1; }
        if (bg != cur) {
          if (gi > 0) tc::mma_commit(qdone);       // previous group's MMAs read its Q
          if (!tc::mbar_wait(qfull, gi & 1, kTimeoutNs)) {
            record_timeout(a, &s_abort);
            break;
          }
          cur = bg;
          ++gi;
        }
        const int s = lt % KS;
        const int buf = lt & 1;
        bool w_ok = tc::mbar_wait(&kfull[s], (lt / KS) & 1, kTimeoutNs);
        if (w_ok && uses[buf] > 0) w_ok = tc::mbar_wait(&acc_free[buf], (uses[buf] - 1) & 1, kTimeoutNs);
        if (!w_ok) {
          record_timeout(a, &s_abort);
          break;
        }
        tc::tc_fence_after();
        const uint32_t kbase = tc::smem_u32(k_s + s * kKTileBytes);
        const uint32_t qbase = tc::smem_u32(q_s);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint64_t ad = tc::smem_desc_sw128(kbase + (k >> 2) * (kKTileBytes / 2) + (k & 3) * 32);
          const uint64_t bd = tc::smem_desc_sw128(qbase + (k >> 2) * (kQChunkBytes / 2) + (k & 3) * 32);
          tc::mma_bf16(tmem + buf * 256, ad, bd, idesc, k > 0 ? 1u : 0u);
        }
        tc::mma_commit(&kempty[s]);
        tc::mma_commit(&acc_full[buf]);
        uses[buf]++;
        --tile;
      }
      tc::mma_commit(done);
      tc::mbar_wait(done, 0, kTimeoutNs);
    }
  } else {
    // ---------------- epilogue: one key per thread and row half ----------------
    // 16 warps: (tile parity set, TMEM lane quarter, row half); the second
    // half hands its partial sums to the first through s_half.
    asm volatile("griddepcontrol.wait;" ::: "memory");   // pass 1's partial statistics
    const int e = warp - 2;
    const int set = (e >> 2) & 1;
    const int half = e >> 3;
    const int quarter = warp & 3;
    const int kl = quarter * 32 + lane;
    int bg = 0, tile = 0;
    if (n_my > 0) locate_pre(s_pre, groups, x1 - 1, bg, tile);
    int cur = -1, gi = 0, use = 0;
    for (int lt = 0; lt < n_my; ++lt) {
      while (tile < 0) { --bg; tile = s_pre[bg + 1] - s_pre[bg] - 1; }
      if (bg != cur) {
        // leaving a group: every warp releases its row info, and the next
        // group's info is written only once all of them have
        bool ok = true;
        if (gi > 0) {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(ifree);
          ok = tc::mbar_wait(ifree, (gi - 1) & 1, kTimeoutNs);
        }
        if (!__all_sync(0xffffffffu, ok)) {
          record_timeout(a, &s_abort);
          break;
        }
        // row info of the new group (-lse2 and query position per row) from
        // pass 1's partial slots; warps 2..9 write one row per lane
        if (e < kRowChunk / 32) {
          const int r = e * 32 + lane;
          float nl = -INFINITY;
          int qp = 0x7fffffff;
          if (r < a.rows) {
            nl = -row_lse2(a, s_pre, groups, bg, r, gridDim.x);
            qp = a.q_pos[(int64_t)(bg / a.Hkv) * a.w + r / a.G];
          }
          reinterpret_cast<float*>(info_s)[r] = nl;
          reinterpret_cast<int*>(info_s)[kRowChunk + r] = qp;
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(ifull);
        }
        if (!__all_sync(0xffffffffu, tc::mbar_wait(ifull, gi & 1, kTimeoutNs))) {
          record_timeout(a, &s_abort);
          break;
        }
        cur = bg;
        ++gi;
      }
      if ((lt & 1) != set) { --tile; continue; }
      const int b = bg / a.Hkv;
      const int s = lt % KS;
      bool w_ok = tc::mbar_wait(&acc_full[set], use & 1, kTimeoutNs);
      if (w_ok && a.causal) w_ok = tc::mbar_wait(&kfull[s], (lt / KS) & 1, kTimeoutNs);
      if (!__all_sync(0xffffffffu, w_ok)) {
        record_timeout(a, &s_abort);
        break;
      }
      tc::tc_fence_after();
      const int kpos = a.causal ? pos_s[s * kKeyTile + kl] : 0;
      const float* lse_s = reinterpret_cast<const float*>(info_s) + half * 128;
      const int* qp_s = reinterpret_cast<const int*>(info_s) + kRowChunk + half * 128;
      bool fast = !a.causal;
      if (a.causal) {
        const int4 q4 = reinterpret_cast<const int4*>(qp_s)[lane];
        int mn = min(min(q4.x, q4.y), min(q4.z, q4.w));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        fast = kpos <= mn;
      }
      float cs0 = 0.f, cs1 = 0.f, cs2 = 0.f, cs3 = 0.f;
      colsum_tile_seq<4>(tmem + ((uint32_t)(quarter * 32) << 16) + set * 256 + half * 128, fast,
                         kpos, lse_s, qp_s, a.scale, cs0, cs1, cs2, cs3);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&acc_free[set]);
        tc::mbar_arrive(&pfree[s]);
      }
      float colsum = (cs0 + cs1) + (cs2 + cs3);
      const int hbuf = use & 1;              // s_half buffer of this tile
      const int hb = set * 2 + hbuf;
      const int k_use = use >> 1;           // earlier uses of this buffer
      ++use;
      if (half == 1) {
        const bool ok = k_use == 0 || tc::mbar_wait(&hempty[hb], (k_use - 1) & 1, kTimeoutNs);
        if (!__all_sync(0xffffffffu, ok)) {
          record_timeout(a, &s_abort);
          break;
        }
        s_half[set][hbuf][kl] = colsum;
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&hfull[hb]);
        --tile;
        continue;
      }
      if (!__all_sync(0xffffffffu, tc::mbar_wait(&hfull[hb], k_use & 1, kTimeoutNs))) {
        record_timeout(a, &s_abort);
        break;
      }
      colsum += s_half[set][hbuf][kl];
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&hempty[hb]);
      const TileGeom tg = TileGeom::make(a, b);
      const int key = tg.base + tile * kKeyTile + kl;
      if (key >= a.out_lo[b] && key < a.out_hi[b] && key >= tg.lo && key < tg.hi &&
          key < a.scores_stride) {
        float* out = a.scores + (int64_t)bg * a.scores_stride + key;
        *out = a.accumulate ? *out + colsum : colsum;
      }
      --tile;
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

constexpr size_t kSmem1 = 1024 + kQChunkBytes + kStages1 * kKTileBytes + kStages1 * kKeyTile * 4 + 256;
constexpr size_t kSmem2 = 1024 + 2 * kQChunkBytes + 2 * kKTileBytes + 4 * kKeyTile * 4 +
                          2 * kRowChunk * 8 + 256;
constexpr size_t kSmem2Resident = 1024 + kQChunkBytes + 4 * kKTileBytes + 4 * kKeyTile * 4 +
                                  kRowChunk * 8 + 256;

struct TcPlan {
  int RC, n_splits, tiles_per_split, tiles_per_cta2, n_tiles_max;
};

TcPlan plan(const se_paged_kv* kv, int w, int n_max) {
  TcPlan p;
  const int G = kv->Hq / kv->Hkv;
  p.RC = cdiv(w * G, kRowChunk);
  // one extra tile when attn_lo is not page aligned
  p.n_tiles_max = cdiv(n_max + kv->page_size, kKeyTile);
  p.tiles_per_split = 16;   // <= kMaxTilesPerSplit
  p.n_splits = cdiv(p.n_tiles_max, p.tiles_per_split);
  p.tiles_per_cta2 = p.RC == 1 ? 16 : 2;
  return p;
}

}  // namespace

bool score_tc_supported(const se_paged_kv* kv) {
  const int G = kv->Hq / kv->Hkv;
  return kv->dtype == SE_BF16 && kv->D == kD && (G == 1 || G == 2 || G == 4 || G == 8) &&
         (kv->page_size == 16 || kv->page_size == 32 || kv->page_size == 64) &&
         (int64_t)kv->num_pages * kv->Hkv * kv->page_size < (int64_t)1 << 31;
}

constexpr int kMaxPersistentCTAs = 256;   // partial slots per row of the persistent pass 1

size_t score_fused_ws(const se_paged_kv* kv, int w, int n_max);
size_t score_fused_ctrl_bytes(const se_paged_kv* kv);
bool score_fused_applicable(const se_paged_kv* kv, int w, int n_max, int n_sm, int smem_optin);
se_status launch_score_fused(const se_paged_kv* kv, const CUtensorMap& kmap, const CUtensorMap& qmap,
                             int w, const int32_t* q_pos, const int32_t* attn_lo,
                             const int32_t* attn_hi, const int32_t* out_lo, const int32_t* out_hi,
                             int causal, int accumulate, int n_max, float* scores,
                             int64_t scores_stride, void* ws, int n_sm, cudaStream_t st);

// Workspace: the one-launch scorer's control block first (it must stay zero
// between calls, so the two-kernel forms carve their buffers after it), then
// the larger of the two forms' buffers.
size_t score_tc_ws(const se_paged_kv* kv, int w, int n_max) {
  const TcPlan p = plan(kv, w, n_max);
  WsCarver c(nullptr);
  c.take<uint8_t>(score_fused_ctrl_bytes(kv));
  const int slots = std::max(2 * p.n_splits, p.RC == 1 ? 2 * kMaxPersistentCTAs : 0);
  c.take<float>((size_t)kv->B * kv->Hkv * p.RC * kRowChunk * slots * 2);
  c.take<float2>((size_t)kv->B * kv->Hkv * p.RC * kRowChunk);
  return std::max(c.bytes(), score_fused_ws(kv, w, n_max));
}

// one_launch: 0 -- the two- or three-launch forms; 1 -- both sweeps in one
// cooperative launch (SE_ERR_UNSUPPORTED when the shape does not allow it).
se_status launch_score_tc(const se_paged_kv* kv, const void* q_win, int w, const int32_t* q_pos,
                          const int32_t* attn_lo, const int32_t* attn_hi, const int32_t* out_lo,
                          const int32_t* out_hi, int causal, int accumulate, int n_max,
                          float* scores, int64_t scores_stride, void* ws, cudaStream_t st,
                          int one_launch) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return SE_ERR_CUDA;
  const int G = kv->Hq / kv->Hkv;
  const TcPlan p = plan(kv, w, n_max);
  CUtensorMap kmap, qmap;
  {
    cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)kv->num_pages * kv->Hkv * kv->page_size};
    cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kv->page_size};
    cuuint32_t estr[2] = {1, 1};
    if (enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv->k_pool, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SE_ERR_CUDA;
  }
  {
    cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)kv->Hq, (cuuint64_t)w, (cuuint64_t)kv->B};
    cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)kv->Hq * kD * 2,
                             (cuuint64_t)w * kv->Hq * kD * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)(kRowChunk / G), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (enc(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q_win), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SE_ERR_CUDA;
  }
  TcArgs a{};
  a.B = kv->B; a.Hq = kv->Hq; a.Hkv = kv->Hkv; a.G = G; a.w = w; a.P = kv->page_size;
  a.rows = w * G; a.RC = p.RC;
  a.max_pages_per_seq = kv->max_pages_per_seq; a.num_pages = kv->num_pages;
  a.block_table = kv->block_table; a.slot_map = kv->slot_map;
  a.smax = (int64_t)kv->max_pages_per_seq * kv->page_size;
  a.q_pos = q_pos; a.attn_lo = attn_lo; a.attn_hi = attn_hi; a.out_lo = out_lo; a.out_hi = out_hi;
  a.causal = causal; a.accumulate = accumulate; a.n_max = n_max;
  a.scores = scores; a.scores_stride = scores_stride;
  WsCarver c(ws);
  // the control block at the start of the workspace: [0, 8) wait limit,
  // [12, 16) the first wait that gave up
  uint8_t* ctrl = c.take<uint8_t>(score_fused_ctrl_bytes(kv));
  a.limit = reinterpret_cast<const unsigned long long*>(ctrl);
  a.diag = reinterpret_cast<unsigned int*>(ctrl + 12);
  const int slots = std::max(2 * p.n_splits, p.RC == 1 ? 2 * kMaxPersistentCTAs : 0);
  a.part = c.take<float>((size_t)kv->B * kv->Hkv * p.RC * kRowChunk * slots * 2);
  a.rowinfo = c.take<float2>((size_t)kv->B * kv->Hkv * p.RC * kRowChunk);
  a.n_splits = p.n_splits; a.tiles_per_split = p.tiles_per_split;
  a.tiles_per_cta2 = p.tiles_per_cta2;
  a.status = kv->status;
  a.scale = kLog2e / sqrtf((float)kD);
  static std::atomic<uint64_t> attr[4];
  if (!allow_smem(reinterpret_cast<const void*>(&score_rowstats_tc), (int)kSmem1, attr[0]) ||
      !allow_smem(reinterpret_cast<const void*>(&score_colsum_tc), (int)kSmem2, attr[1]) ||
      !allow_smem(reinterpret_cast<const void*>(&score_colsum_persistent_tc), (int)kSmem2Resident,
                  attr[2]) ||
      !allow_smem(reinterpret_cast<const void*>(&score_rowstats_persistent_tc), (int)kSmem1,
                  attr[3]))
    return SE_ERR_CUDA;
  const int groups = kv->B * kv->Hkv;
  int dev = 0, n_sm = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return SE_ERR_CUDA;
  if (one_launch) {
    // both passes in one cooperative launch, every key read from HBM once
    if (!score_fused_applicable(kv, w, n_max, n_sm, optin)) return SE_ERR_UNSUPPORTED;
    return launch_score_fused(kv, kmap, qmap, w, q_pos, attn_lo, attn_hi, out_lo, out_hi, causal,
                              accumulate, n_max, scores, scores_stride, ws, n_sm, st);
  }
  if (p.RC == 1 && groups <= kMaxGroupsP) {
    // one row chunk: persistent CTAs, one per SM, over the (group, tile) sequence
    const int ctas = std::min(std::min(n_sm, kMaxPersistentCTAs), groups * p.n_tiles_max);
    se_launch(score_rowstats_persistent_tc, ctas, kThreads, kSmem1, st, kmap, qmap, a);
    se_launch(score_colsum_persistent_tc, ctas, kThreads, kSmem2Resident, st, kmap, qmap, a);
    return SE_OK;
  }
  se_launch(score_rowstats_tc, dim3(p.n_splits, p.RC, groups), kThreads, kSmem1, st, kmap, qmap, a);
  se_launch(score_rowinfo_tc, dim3(cdiv(p.RC * kRowChunk, 256), groups), 256, 0, st, a);
  se_launch(score_colsum_tc, dim3(cdiv(p.n_tiles_max, p.tiles_per_cta2), groups), kThreads, kSmem2, st,
      kmap, qmap, a);
  return SE_OK;
}

}  // namespace se
