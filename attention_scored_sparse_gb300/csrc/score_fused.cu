// Window scoring in one cooperative launch that reads every key from HBM once
// (bf16, D = 128, at most 256 rows -- window queries x heads of a group).
//
// SparseEngine "How it works" (SnapKV / H2O: attention of the window queries
// over the cached keys) and KARA Method 1:
//     s[b, g, j] = sum_{h in g} sum_{q in window} softmax_j(q . k_j / sqrt(D))
// A row's softmax needs its whole row before a column can be summed, so every
// key tile is visited twice: pass 1 (row statistics, rows on TMEM lanes) and
// pass 2 (column sums, keys on TMEM lanes).  The two-kernel form reads the
// keys from HBM twice; here both passes run in one grid of one CTA per SM
// and pass 2 of a key tile follows pass 1 of the same tile closely enough
// that the tile is still in L2.
//
// Work order.  The (group, key tile) sequence is cut into W waves at group
// boundaries, each small enough that three waves fit in L2; within a wave
// CTA c takes the c-th contiguous share of the tiles (its segment).  Every
// CTA walks its segments in the order
//     P1(0) P1(1) P1(2) P2(0) P1(3) P2(1) ... P1(W-1) P2(W-3) P2(W-2) P2(W-1)
// (pass 2 of a wave two waves behind pass 1), reading the keys of pass 1
// with an evict-last and those of pass 2 with an evict-first L2 policy.
//
// Row statistics across CTAs.  Pass 1 keeps, per row and column half, a
// base-2 running (max, sum) over the CTA's tiles of a group and writes it to
// a partial slot at the end of its context (a run of tiles of one group and
// pass).  A bookkeeping warp counts the context's tiles into the group's
// counter (device-scope fence, atomic add) and merges partial slots: the
// rows of a group are shared out among the CTAs that hold its tiles, in
// proportion to their tiles, and each CTA merges its rows one segment before
// it needs them (at its pass-2 segment of the previous wave), once the
// group's counter shows every tile counted.  A merged row is one 64-bit word
// -- -log2 of the row's softmax denominator and a tag for this call -- so a
// pass-2 context only checks the tags of its group's rows (bounded wait) and
// no fence or flag is needed between the rows and their readers.  Every CTA
// is resident for the whole launch (cooperative launch), so these waits end;
// each is bounded by %globaltimer and on expiry sets SE_ERR_TIMEOUT and the
// launch winds down.  The CTA that takes a wave's i-th share rotates from
// wave to wave, so the spare tiles of uneven shares spread over the CTAs.
//
// Pass 1 with a stale maximum: the running maximum of a row is taken from
// the first tile of a context; later tiles add exp2(x - m) to the sum
// without a maximum and only recompute when a tile's sum grows past 2^64
// (a logit more than ~58 above m), so the common tile costs one FFMA2, two
// exp2 and one FADD2 per two logits.  The sum is exact up to rounding for
// any m below the true maximum; m stays a logit of the row, so the sum is at
// least 1 and nothing it keeps underflows.
//
// Roles (19 warps): warp 0 TMA producer, warp 1 MMA issuer, warp 2
// bookkeeper, warps 3..18 epilogue (four per TMEM lane quarter).  Q is
// double-buffered (the next context's Q loads while the current one is in
// use), K runs through three stages.
#include <cuda.h>

#include <algorithm>

#include "tc_primitives.cuh"

namespace se {

namespace {

constexpr int kD = 128;
constexpr int kKeyTile = 128;
constexpr int kRows = 256;
constexpr int kKTileBytes = kKeyTile * kD * 2;   // 32 KB
constexpr int kQBytes = kRows * kD * 2;          // 64 KB
constexpr int kQS = 2;                           // Q buffers
constexpr int kKS = 3;                           // K stages
constexpr int kEpiWarps = 16;
constexpr int kEpi0 = 3;                         // first epilogue warp
constexpr int kWarps = kEpi0 + kEpiWarps;
constexpr int kThreads = kWarps * 32;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kRing = 16;                        // pass-1 contexts between epilogue and bookkeeper
constexpr int kMaxB = 128;                       // sequences indexed in shared memory
constexpr int kMaxCTAs = 256;
constexpr uint64_t kLimitNs = 2000000000ull;     // 2 s per wait
constexpr float kGuard = 18446744073709551616.0f;   // 2^64

// Control block at the start of the workspace: zero before the first call.
// [0, 8): optional wait limit in ns (0 = 2 s); [8, 12): CTAs finished (back
// to 0 after each call); [12, 16): where the first bounded wait that gave up
// was (site | warp << 8 | CTA << 16, plus 1; for the caller to read and
// clear); [16, 20): calls so far (tags the merged rows of each call); from
// byte 64, per group the pass-1 tile counter (back to 0 after each call).
constexpr int kCtrlHead = 64;
constexpr int kRot = 53;                         // share rotation from wave to wave

struct FusedArgs {
  int B, Hq, Hkv, G, w, P, rows, groups;
  int max_pages_per_seq;
  const int32_t* block_table;
  const int32_t* slot_map;
  int64_t smax;
  const int32_t* q_pos;
  const int32_t* attn_lo;
  const int32_t* attn_hi;
  const int32_t* out_lo;
  const int32_t* out_hi;
  int causal, accumulate, n_max;
  float* scores;
  int64_t scores_stride;
  const unsigned long long* limit_override;
  unsigned int* exit_count;
  unsigned int* diag;
  unsigned int* epoch;
  unsigned int* cnt;       // [groups]
  unsigned long long* rowinfo;  // [groups][256]: -lse2 bits | tag << 32
  float2* part;            // [slots][256 rows][2 halves] (max, sum)
  int W;
  int32_t* status;
  float scale;             // log2(e) / sqrt(D)
};

// Shared memory: Q buffers and K stages (1024-byte aligned for the 128-byte
// swizzle), then barriers and small tables.
struct __align__(8) Bars {
  uint64_t kfull[kKS], kempty[kKS];
  uint64_t qfull[kQS], qfree[kQS];
  uint64_t acc_full[2], acc_free[2];
  uint64_t p1d[kRing], p1e[kRing];
  uint64_t done;
  uint32_t tmem;
  int abort_flag;
  int Hkv, groups, W;      // geometry read by the work-order helpers
  int seq_pre[kMaxB + 1];  // key tiles of sequences 0 .. b-1 (all their groups)
  int seq_nt[kMaxB];       // key tiles of one group of sequence b
};

constexpr size_t kTileBytes = (size_t)kQS * kQBytes + (size_t)kKS * kKTileBytes;
constexpr size_t kSmemBytes = 1024 + kTileBytes + sizeof(Bars);
static_assert(kSmemBytes <= 232448, "one CTA per SM: at most 227 KB of shared memory");

SE_DEV bool aborted(const int* f) { return *reinterpret_cast<const volatile int*>(f) != 0; }

// Sites of the bounded waits, for the diagnostic word.
enum : unsigned { kAtQfree = 1, kAtKempty, kAtQfull, kAtKfull, kAtP1d, kAtCount, kAtRows,
                  kAtAccFull, kAtP1e };

SE_DEV void record_timeout(const FusedArgs& a, int* abort_flag, unsigned site) {
  set_status(a.status, SE_ERR_TIMEOUT);
  atomicCAS(a.diag, 0u, 1u + (site | (threadIdx.x >> 5) << 8 | blockIdx.x << 16));
  atomicExch(abort_flag, 1);
}

SE_DEV uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

SE_DEV uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

SE_DEV void tma_load_2d_hint(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_u32(bar)), "l"(policy)
      : "memory");
}

SE_DEV void tmem_st1(uint32_t taddr, float v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr),
               "r"(__float_as_uint(v))
               : "memory");
}

SE_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

SE_DEV void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

SE_DEV unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

SE_DEV unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

SE_DEV ulonglong2 ld_u2(const unsigned long long* p) {
  ulonglong2 v;
  asm volatile("ld.global.v2.u64 {%0, %1}, [%2];" : "=l"(v.x), "=l"(v.y) : "l"(p));
  return v;
}

SE_DEV float2 ld_cg_f2(const float2* p) {
  float2 v;
  asm volatile("ld.global.cg.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------
// Work order shared by every role.
// ---------------------------------------------------------------------------

// Pass and wave of the k-th segment of a CTA's list (2W segments).
SE_DEV void seg_kind(int k, int W, int& pass, int& wave) {
  if (W <= 2) {
    pass = k < W ? 1 : 2;
    wave = k < W ? k : k - W;
    return;
  }
  if (k < 2) { pass = 1; wave = k; return; }
  if (k >= 2 * W - 2) { pass = 2; wave = k - W; return; }
  if ((k & 1) == 0) { pass = 1; wave = k / 2 + 1; } else { pass = 2; wave = (k - 3) / 2; }
}

// Work-order geometry; its sizes live in shared memory and the CTA count is
// the grid's, so a copy costs one register.
struct Geo {
  const Bars* s;
  SE_DEV int Hkv() const { return s->Hkv; }
  SE_DEV int groups() const { return s->groups; }
  SE_DEV int W() const { return s->W; }
  SE_DEV int C() const { return (int)gridDim.x; }
  SE_DEV int group_start(int gi) const {   // global index of group gi's first tile
    if (gi >= groups()) return s->seq_pre[groups() / Hkv()];
    const int b = gi / Hkv();
    return s->seq_pre[b] + (gi % Hkv()) * s->seq_nt[b];
  }
  SE_DEV int wave_group(int w) const { return (int)((int64_t)w * groups() / W()); }
  SE_DEV int wave_of(int gi) const { return (int)(((int64_t)(gi + 1) * W() - 1) / groups()); }
  // Share i of wave w (shares are contiguous tile ranges, i = 0 .. C-1).
  SE_DEV void share_range(int w, int i, int& x0, int& x1) const {
    const int t0 = group_start(wave_group(w)), t1 = group_start(wave_group(w + 1));
    const int64_t n = t1 - t0;
    x0 = t0 + (int)((int64_t)i * n / C());
    x1 = t0 + (int)((int64_t)(i + 1) * n / C());
  }
  // The share CTA c takes in wave w, and its tiles.
  SE_DEV int share_of(int w, int c) const { return (int)(((int64_t)c + (int64_t)w * kRot) % C()); }
  SE_DEV void seg_range(int w, int c, int& x0, int& x1) const { share_range(w, share_of(w, c), x0, x1); }
  // Segment (w * C + share) holding tile x of group gi.
  SE_DEV int seg_of(int gi, int x) const {
    const int w = wave_of(gi);
    const int t0 = group_start(wave_group(w)), t1 = group_start(wave_group(w + 1));
    const int64_t n = t1 - t0;
    const int i = (int)(((int64_t)(x - t0 + 1) * C() - 1) / n);
    return w * C() + i;
  }
  // Group and tile within the group of global tile x (x below the total).
  SE_DEV void locate(int x, int& gi, int& tile) const {
    const int B = groups() / Hkv();
    int lo = 0, hi = B;                   // largest b with seq_pre[b] <= x
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s->seq_pre[mid] <= x) lo = mid; else hi = mid;
    }
    int b = lo;
    while (b < B - 1 && s->seq_pre[b + 1] <= x) ++b;
    const int off = x - s->seq_pre[b];
    gi = b * Hkv() + off / s->seq_nt[b];
    tile = off % s->seq_nt[b];
  }
};

// Walks the CTA's (segment, tile) items in order.
struct Walk {
  Geo geo;
  int k;            // segment index in the CTA's list
  int pass, wave;
  int x, x1;        // current tile (global index) and segment end
  int gi, tile;     // current group and tile within it
  int ctx;          // context number (0-based) of the current item
  bool valid;
  SE_DEV void start_segment() {
    while (k < 2 * geo.W()) {
      seg_kind(k, geo.W(), pass, wave);
      geo.seg_range(wave, blockIdx.x, x, x1);
      if (x < x1) {
        geo.locate(x, gi, tile);
        return;
      }
      ++k;
    }
    valid = false;
  }
  SE_DEV void init(const Geo& g) {
    geo = g;
    k = 0;
    pass = 1;
    wave = 0;
    x = x1 = 0;
    gi = tile = 0;
    ctx = 0;
    valid = true;
    start_segment();
  }
  // Number of tiles left in the current context, this one included.
  SE_DEV int left_in_context() const { return min(x1, geo.group_start(gi + 1)) - x; }
  SE_DEV void next() {
    const int left = left_in_context();
    ++x;
    ++tile;
    if (x >= x1) {
      ++k;
      ++ctx;
      start_segment();
      return;
    }
    if (left == 1) {          // crossed into the next group of the segment
      ++ctx;
      geo.locate(x, gi, tile);
    }
  }
};

// ---------------------------------------------------------------------------
// Loads
// ---------------------------------------------------------------------------

SE_DEV void load_q(const FusedArgs& a, const CUtensorMap* qmap, int gi, uint8_t* dst,
                   uint64_t* bar) {
  const int b = gi / a.Hkv, g = gi % a.Hkv;
  tc::mbar_arrive_expect_tx(bar, kQBytes);
  tc::tma_load_4d(dst, qmap, bar, 0, g * a.G, 0, b);
  tc::tma_load_4d(dst + kQBytes / 2, qmap, bar, 64, g * a.G, 0, b);
}

// The pages of key tile `tile` of group gi (their row coordinate in the key
// map; np of them, the rest -1), read from the block table with independent
// loads so that one latency covers them all.
struct TilePages {
  int y[kKeyTile / 16];
  int np;
};

SE_DEV TilePages tile_pages(const FusedArgs& a, int gi, int tile) {
  TilePages t;
  const int b = gi / a.Hkv, g = gi % a.Hkv;
  const int P = a.P;
  const int base = (a.attn_lo[b] / P) * P;
  const int end_block = cdiv(a.attn_hi[b], P);
  const int blk0 = base / P + tile * (kKeyTile / P);
  t.np = max(0, min(kKeyTile / P, end_block - blk0));
  const int32_t* bt = a.block_table + (int64_t)b * a.max_pages_per_seq + blk0;
#pragma unroll
  for (int i = 0; i < kKeyTile / 16; ++i) t.y[i] = i < t.np ? bt[i] : -1;
#pragma unroll
  for (int i = 0; i < kKeyTile / 16; ++i) t.y[i] = (t.y[i] * a.Hkv + g) * P;
  return t;
}

SE_DEV void load_k(const FusedArgs& a, const TilePages& t, const CUtensorMap* kmap, uint8_t* dst,
                   uint64_t* bar, uint64_t policy) {
  const int P = a.P;
  tc::mbar_arrive_expect_tx(bar, (uint32_t)t.np * P * kD * 2);
#pragma unroll
  for (int i = 0; i < kKeyTile / 16; ++i) {
    if (i < t.np) {
      tma_load_2d_hint(dst + i * P * 128, kmap, bar, 0, t.y[i], policy);
      tma_load_2d_hint(dst + kKTileBytes / 2 + i * P * 128, kmap, bar, 64, t.y[i], policy);
    }
  }
}

// ---------------------------------------------------------------------------
// Epilogue pieces
// ---------------------------------------------------------------------------

// Pass-1 update of one row's (m, l) with a block of N logits, every one of
// them in range and visible.  m = -inf: first block of the context.
template <int N>
SE_DEV void p1_fast(const uint32_t (&r)[N], float scale, float& m, float& l) {
  if (m == -INFINITY) {
    float c0 = __uint_as_float(r[0]), c1 = __uint_as_float(r[1]);
#pragma unroll
    for (int j = 2; j < N; j += 4) {
      c0 = tc::fmax3(c0, __uint_as_float(r[j]), __uint_as_float(r[j + 1]));
      c1 = tc::fmax3(c1, __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
    }
    m = fmaxf(c0, c1) * scale;
  }
  const uint64_t sc2 = tc::f2(scale, scale);
  const uint64_t nm2 = tc::f2(-m, -m);
  uint64_t s0 = 0, s1 = 0, s2 = 0, s3 = 0;
#pragma unroll
  for (int j = 0; j < N; j += 8) {
    float a0, a1, b0, b1, c0, c1, d0, d1;
    tc::f2split(tc::ffma2(tc::f2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), sc2, nm2), a0, a1);
    tc::f2split(tc::ffma2(tc::f2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])), sc2, nm2), b0, b1);
    tc::f2split(tc::ffma2(tc::f2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5])), sc2, nm2), c0, c1);
    tc::f2split(tc::ffma2(tc::f2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7])), sc2, nm2), d0, d1);
    s0 = tc::fadd2(s0, tc::f2(tc::ex2(a0), tc::ex2(a1)));
    s1 = tc::fadd2(s1, tc::f2(tc::ex2(b0), tc::ex2(b1)));
    s2 = tc::fadd2(s2, tc::f2(tc::ex2(c0), tc::ex2(c1)));
    s3 = tc::fadd2(s3, tc::f2(tc::ex2(d0), tc::ex2(d1)));
  }
  float x0, x1, y0, y1, z0, z1, w0, w1;
  tc::f2split(s0, x0, x1);
  tc::f2split(s1, y0, y1);
  tc::f2split(s2, z0, z1);
  tc::f2split(s3, w0, w1);
  const float t = ((x0 + x1) + (y0 + y1)) + ((z0 + z1) + (w0 + w1));
  if (t <= kGuard) {
    l += t;
    return;
  }
  // a logit far above m: redo the block with its own maximum
  float c0 = -INFINITY;
#pragma unroll
  for (int j = 0; j < N; ++j) c0 = fmaxf(c0, __uint_as_float(r[j]));
  const float mn = fmaxf(m, c0 * scale);
  float u = 0.f;
#pragma unroll
  for (int j = 0; j < N; ++j) u += tc::ex2(fmaf(__uint_as_float(r[j]), scale, -mn));
  l = l * tc::ex2(m - mn) + u;
  m = mn;
}

// Pass-1 update with a per-column visibility mask (range ends, causal) for
// columns [col0, col0 + N) of the warp's 64; lane i holds the positions of
// columns 2i and 2i+1 in pos2.  Every lane runs every shuffle.
template <int N>
SE_DEV void p1_masked(const uint32_t (&r)[N], int col0, int2 pos2, bool row_ok, int key0, int lo,
                      int hi, bool causal, int qpos, float scale, float& m, float& l) {
  float cm = -INFINITY;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const int c = col0 + j;
    const int pj = __shfl_sync(0xffffffffu, (c & 1) ? pos2.y : pos2.x, c >> 1);
    const int key = key0 + c;
    const bool vis = row_ok && key >= lo && key < hi && (!causal || pj <= qpos);
    if (vis) cm = fmaxf(cm, __uint_as_float(r[j]) * scale);
  }
  const float mn = fmaxf(m, cm);
  float u = 0.f;
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const int c = col0 + j;
    const int pj = __shfl_sync(0xffffffffu, (c & 1) ? pos2.y : pos2.x, c >> 1);
    const int key = key0 + c;
    const bool vis = row_ok && key >= lo && key < hi && (!causal || pj <= qpos);
    if (vis) u += tc::ex2(fmaf(__uint_as_float(r[j]), scale, -mn));
  }
  if (cm == -INFINITY) return;   // nothing of this block is visible to the row
  l = (m == -INFINITY ? 0.f : l * tc::ex2(m - mn)) + u;
  m = mn;
}

// Pass-2 column sum of one key over a block of N rows r0 .. r0+N-1:
// exp2(x * scale - lse2_row).  rows: the tagged -lse2 words of the block
// (global, read through L1); qrow: query positions of the sequence (read
// only when masked; row r belongs to query r / G).
template <int N>
SE_DEV float p2_sum(const uint32_t (&r)[N], const unsigned long long* rows, const int* qrow, int r0,
                    int n_rows, int G, bool masked, int kpos, float scale) {
  const uint64_t sc2 = tc::f2(scale, scale);
  uint64_t s0 = 0, s1 = 0;
  if (!masked) {
#pragma unroll
    for (int j = 0; j < N; j += 4) {
      const ulonglong2 n01 = ld_u2(rows + j), n23 = ld_u2(rows + j + 2);
      float a0, a1, b0, b1;
      tc::f2split(tc::ffma2(tc::f2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), sc2,
                            tc::f2(__uint_as_float((uint32_t)n01.x), __uint_as_float((uint32_t)n01.y))),
                  a0, a1);
      tc::f2split(tc::ffma2(tc::f2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])), sc2,
                            tc::f2(__uint_as_float((uint32_t)n23.x), __uint_as_float((uint32_t)n23.y))),
                  b0, b1);
      s0 = tc::fadd2(s0, tc::f2(tc::ex2(a0), tc::ex2(a1)));
      s1 = tc::fadd2(s1, tc::f2(tc::ex2(b0), tc::ex2(b1)));
    }
  } else {
#pragma unroll 4
    for (int j = 0; j < N; ++j) {
      const int row = r0 + j;
      const int qp = row < n_rows ? qrow[row / G] : 0x7fffffff;
      const float n = __uint_as_float((uint32_t)rows[j]);
      float p = tc::ex2(fmaf(__uint_as_float(r[j]), scale, n));
      if (kpos > qp) p = 0.f;
      s0 = tc::fadd2(s0, tc::f2(p, 0.f));
    }
  }
  float x0, x1, y0, y1;
  tc::f2split(s0, x0, x1);
  tc::f2split(s1, y0, y1);
  return (x0 + x1) + (y0 + y1);
}

// Three single columns of the warp's TMEM lanes, one wait.
SE_DEV void tmem_ld3(uint32_t t0, uint32_t t1, uint32_t t2, float& a, float& b, float& c) {
  uint32_t x, y, z;
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%3];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%1}, [%4];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x1.b32 {%2}, [%5];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(x), "=r"(y), "=r"(z)
      : "r"(t0), "r"(t1), "r"(t2)
      : "memory");
  a = __uint_as_float(x);
  b = __uint_as_float(y);
  c = __uint_as_float(z);
}

// Merge of rows [r0, r1) of group gi from its partial slots into tagged
// -lse2 words (one warp; lanes share out the slots of four rows at a time).
SE_DEV void merge_rows(const FusedArgs& a, const Geo& geo, int gi, int r0, int r1,
                       unsigned long long tag, int lane) {
  const int x0 = geo.group_start(gi), x1 = geo.group_start(gi + 1);
  const int s0 = geo.seg_of(gi, x0), s1 = geo.seg_of(gi, x1 - 1);   // segments (w * C + share)
  const int C = geo.C();
  const int w = s0 / C, i0 = s0 % C;
  // shares of this wave with no tiles (more CTAs than tiles) wrote no slot
  const int t0 = geo.group_start(geo.wave_group(w)), t1 = geo.group_start(geo.wave_group(w + 1));
  const int n = t1 - t0;
  const bool all_full = n >= C;
  const int n_ent = (s1 - s0 + 1) * 2;
  for (int rb = r0; rb < r1; rb += 4) {
    float M[4], L[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) { M[u] = -INFINITY; L[u] = 0.f; }
    for (int e0 = 0; e0 < n_ent; e0 += 128) {
      float2 v[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = e0 + q * 32 + lane;
        const int sh = i0 + (e >> 1);                     // share index within wave w
        bool ok = e < n_ent;
        if (ok && !all_full)
          ok = (int)((int64_t)(sh + 1) * n / C) > (int)((int64_t)sh * n / C);
        const float2* src = a.part + ((int64_t)(s0 + (e >> 1) + gi) * kRows) * 2 + (e & 1);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = rb + u;
          v[u][q] = ok && r < r1 && r < a.rows ? ld_cg_f2(src + r * 2) : make_float2(-INFINITY, 0.f);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float m = v[u][q].x;
          const float mx = fmaxf(M[u], m);
          if (mx == -INFINITY) continue;
          L[u] = L[u] * tc::ex2(M[u] - mx) + v[u][q].y * tc::ex2(m - mx);
          M[u] = mx;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float Mo = __shfl_xor_sync(0xffffffffu, M[u], o);
        const float Lo = __shfl_xor_sync(0xffffffffu, L[u], o);
        const float Mx = fmaxf(M[u], Mo);
        if (Mx != -INFINITY) {
          L[u] = L[u] * tc::ex2(M[u] - Mx) + Lo * tc::ex2(Mo - Mx);
          M[u] = Mx;
        }
      }
      const int r = rb + u;
      if (lane == 0 && r < r1) {
        const float nl = r < a.rows && L[u] > 0.f ? -(M[u] + log2f(L[u])) : -INFINITY;
        a.rowinfo[(int64_t)gi * kRows + r] = (unsigned long long)__float_as_uint(nl) | (tag << 32);
      }
    }
  }
}

// Merges this CTA's share of the rows of every group that its tiles of wave
// w meet, once each group's pass-1 tiles are all counted (one warp).
SE_DEV bool merge_wave(const FusedArgs& a, const Geo& geo, int w, int c, unsigned long long tag,
                       uint64_t limit, int* abort_flag, int lane) {
  int x0, x1;
  geo.seg_range(w, c, x0, x1);
  int x = x0;
  while (x < x1) {
    int gi, t;
    geo.locate(x, gi, t);
    const int gs = geo.group_start(gi), ge = geo.group_start(gi + 1);
    const int xe = min(x1, ge);
    const int nt = ge - gs;
    bool ok = true;
    if (lane == 0) {
      if (ld_acquire(&a.cnt[gi]) != (unsigned)nt) {
        const uint64_t t0 = tc::globaltimer();
        while (ld_acquire(&a.cnt[gi]) != (unsigned)nt) {
          if (aborted(abort_flag) || tc::globaltimer() - t0 > limit) { ok = false; break; }
        }
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    if (!ok) return false;
    const int r0 = (int)((int64_t)(x - gs) * kRows / nt), r1 = (int)((int64_t)(xe - gs) * kRows / nt);
    merge_rows(a, geo, gi, r0, r1, tag, lane);
    x = xe;
  }
  return true;
}

}  // namespace

// ---------------------------------------------------------------------------
// The kernel.  grid = C CTAs (cooperative), 608 threads.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 1)
score_fused_tc(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
               FusedArgs a) {
  pdl_enter();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* q_s = smem;                              // [kQS][64 KB]
  uint8_t* k_s = q_s + kQS * kQBytes;               // [kKS][32 KB]
  Bars* s = reinterpret_cast<Bars*>(k_s + kKS * kKTileBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t limit =
      a.limit_override != nullptr && *a.limit_override != 0 ? *a.limit_override : kLimitNs;

  // per-sequence tile geometry (every CTA computes the same tables)
  const int B = a.B;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int lo = a.attn_lo[b], hi = a.attn_hi[b];
    const bool ok = lo >= 0 && hi >= lo && hi - lo <= a.n_max && (int64_t)hi <= a.smax;
    const int base = (lo / a.P) * a.P;
    s->seq_nt[b] = ok && hi > lo ? cdiv(hi - base, kKeyTile) : 0;
    if (!ok) set_status(a.status, SE_ERR_BOUNDS);
  }
  if (threadIdx.x == 0) {
    s->abort_flag = 0;
    s->Hkv = a.Hkv;
    s->groups = a.groups;
    s->W = a.W;
    for (int i = 0; i < kKS; ++i) {
      tc::mbar_init(&s->kfull[i], 1);
      tc::mbar_init(&s->kempty[i], 1);
    }
    for (int i = 0; i < kQS; ++i) {
      tc::mbar_init(&s->qfull[i], 1);
      tc::mbar_init(&s->qfree[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(&s->acc_full[i], 1);
      tc::mbar_init(&s->acc_free[i], kEpiWarps);
    }
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(&s->p1d[i], kEpiThreads);
      tc::mbar_init(&s->p1e[i], 1);
    }
    tc::mbar_init(&s->done, 1);
    tc::fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&s->tmem, 512);
  __syncthreads();
  if (threadIdx.x == 0) {
    int acc = 0;
    for (int b = 0; b < B; ++b) {
      s->seq_pre[b] = acc;
      acc += a.Hkv * s->seq_nt[b];
    }
    s->seq_pre[B] = acc;
  }
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = s->tmem;
  Geo geo{s};
  // tag of this call's merged rows (never zero, so a zeroed workspace is not ready)
  const unsigned long long tag = (unsigned long long)((*a.epoch & 0x7fffffffu) | 0x80000000u);

  if (warp == 0) {
    // ---------------- producer ----------------
    if (tc::elect_one()) {
      tc::tma_prefetch_desc(&kmap);
      tc::tma_prefetch_desc(&qmap);
      const uint64_t pol1 = policy_evict_last(), pol2 = policy_evict_first();
      Walk wk;
      wk.init(geo);
      int i = 0, q_issued = 0;   // K tiles and Q contexts issued
      int cur_ctx = -1;
      // lookahead walker: the context after the current one, for the Q prefetch
      Walk ahead = wk;
      bool stop = false;
      TilePages pages{};                                  // read a tile ahead
      if (wk.valid) pages = tile_pages(a, wk.gi, wk.tile);
      while (wk.valid && !stop && !aborted(&s->abort_flag)) {
        if (wk.ctx != cur_ctx) {
          cur_ctx = wk.ctx;
          // Q of this context (prefetched unless it is the first)
          while (q_issued <= cur_ctx) {
            // find the group of context q_issued
            while (ahead.valid && ahead.ctx < q_issued) ahead.next();
            if (!ahead.valid) break;
            const int qb = q_issued % kQS;
            if (q_issued >= kQS &&
                !tc::mbar_wait(&s->qfree[qb], ((q_issued / kQS) - 1) & 1, limit)) {
              record_timeout(a, &s->abort_flag, kAtQfree);
              stop = true;
              break;
            }
            load_q(a, &qmap, ahead.gi, q_s + qb * kQBytes, &s->qfull[qb]);
            ++q_issued;
          }
          if (stop) break;
        }
        // prefetch the next context's Q once its buffer is free (no wait)
        if (q_issued == cur_ctx + 1) {
          while (ahead.valid && ahead.ctx < q_issued) ahead.next();
          if (ahead.valid) {
            const int qb = q_issued % kQS;
            if (q_issued < kQS || tc::mbar_test_wait(&s->qfree[qb], ((q_issued / kQS) - 1) & 1)) {
              load_q(a, &qmap, ahead.gi, q_s + qb * kQBytes, &s->qfull[qb]);
              ++q_issued;
            }
          }
        }
        const int st = i % kKS;
        if (i >= kKS && !tc::mbar_wait(&s->kempty[st], ((i / kKS) - 1) & 1, limit)) {
          record_timeout(a, &s->abort_flag, kAtKempty);
          break;
        }
        load_k(a, pages, &kmap, k_s + st * kKTileBytes, &s->kfull[st], wk.pass == 1 ? pol1 : pol2);
        ++i;
        wk.next();
        if (wk.valid) pages = tile_pages(a, wk.gi, wk.tile);
      }
      // drain: every issued copy lands before the CTA exits
      for (int j = max(0, i - kKS); j < i; ++j)
        tc::mbar_wait(&s->kfull[j % kKS], (j / kKS) & 1, kLimitNs);
      for (int j = max(0, q_issued - kQS); j < q_issued; ++j)
        tc::mbar_wait(&s->qfull[j % kQS], (j / kQS) & 1, kLimitNs);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (tc::elect_one()) {
      const uint32_t id1 = tc::idesc_bf16_f32(128, kKeyTile);
      const uint32_t id2 = tc::idesc_bf16_f32(128, kRows);
      Walk wk;
      wk.init(geo);
      int i = 0, cur_ctx = -1;
      while (wk.valid && !aborted(&s->abort_flag)) {
        if (wk.ctx != cur_ctx) {
          if (cur_ctx >= 0) tc::mma_commit(&s->qfree[cur_ctx % kQS]);
          cur_ctx = wk.ctx;
          if (!tc::mbar_wait(&s->qfull[cur_ctx % kQS], (cur_ctx / kQS) & 1, limit)) {
            record_timeout(a, &s->abort_flag, kAtQfull);
            break;
          }
        }
        const int st = i % kKS, buf = i & 1;
        if (!tc::mbar_wait(&s->kfull[st], (i / kKS) & 1, limit) ||
            (i >= 2 && !tc::mbar_wait(&s->acc_free[buf], ((i >> 1) - 1) & 1, limit))) {
          record_timeout(a, &s->abort_flag, kAtKfull);
          break;
        }
        tc::tc_fence_after();
        const uint32_t kb = tc::smem_u32(k_s + st * kKTileBytes);
        const uint32_t qb = tc::smem_u32(q_s + (cur_ctx % kQS) * kQBytes);
        if (wk.pass == 1) {
#pragma unroll
          for (int mb = 0; mb < 2; ++mb) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint64_t ad = tc::smem_desc_sw128(qb + (k >> 2) * (kQBytes / 2) + mb * (128 * 128) +
                                                      (k & 3) * 32);
              const uint64_t bd = tc::smem_desc_sw128(kb + (k >> 2) * (kKTileBytes / 2) + (k & 3) * 32);
              tc::mma_bf16(tmem + buf * 256 + mb * 128, ad, bd, id1, k > 0 ? 1u : 0u);
            }
          }
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t ad = tc::smem_desc_sw128(kb + (k >> 2) * (kKTileBytes / 2) + (k & 3) * 32);
            const uint64_t bd = tc::smem_desc_sw128(qb + (k >> 2) * (kQBytes / 2) + (k & 3) * 32);
            tc::mma_bf16(tmem + buf * 256, ad, bd, id2, k > 0 ? 1u : 0u);
          }
        }
        tc::mma_commit(&s->kempty[st]);
        tc::mma_commit(&s->acc_full[buf]);
        ++i;
        wk.next();
      }
      tc::mma_commit(&s->done);
      tc::mbar_wait(&s->done, 0, kLimitNs);
    }
  } else if (warp == 2) {
    // ---------------- bookkeeper: pass-1 tile counts, row merges ----------------
    // Walks the CTA's segments in order: at each pass-1 context end, counts
    // its tiles into the group; at the start of pass-2 segment v, merges
    // this CTA's rows of the groups of wave v + 1 (and of wave 0 at v = 0).
    int j = 0;   // pass-1 contexts
    bool stop = false;
    for (int k = 0; k < 2 * a.W && !stop && !aborted(&s->abort_flag); ++k) {
      int pass, wave;
      seg_kind(k, a.W, pass, wave);
      if (pass == 1) {
        int x0, x1;
        geo.seg_range(wave, blockIdx.x, x0, x1);
        int x = x0;
        while (x < x1) {
          int gi, t;
          geo.locate(x, gi, t);
          const int xe = min(x1, geo.group_start(gi + 1));
          if (lane == 0) {
            if (!tc::mbar_wait(&s->p1d[j % kRing], (j / kRing) & 1, limit)) {
              record_timeout(a, &s->abort_flag, kAtP1d);
            } else {
              __threadfence();
              atomicAdd(&a.cnt[gi], (unsigned)(xe - x));
              tc::mbar_arrive(&s->p1e[j % kRing]);
            }
          }
          __syncwarp();
          if (aborted(&s->abort_flag)) { stop = true; break; }
          ++j;
          x = xe;
        }
      } else {
        bool ok = true;
        if (wave == 0) ok = merge_wave(a, geo, 0, blockIdx.x, tag, limit, &s->abort_flag, lane);
        if (ok && wave + 1 <= a.W - 1)
          ok = merge_wave(a, geo, wave + 1, blockIdx.x, tag, limit, &s->abort_flag, lane);
        if (!ok) {
          if (lane == 0 && !aborted(&s->abort_flag)) record_timeout(a, &s->abort_flag, kAtCount);
          stop = true;
        }
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int e = warp - kEpi0;            // 0..15
    const int quarter = warp & 3;          // TMEM lanes this warp may read
    const int idx = e >> 2;                // pass 1: (mb, half); pass 2: row quarter
    const int mb = idx & 1, half = idx >> 1;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int r = mb * 128 + quarter * 32 + lane;   // pass-1 row of this thread
    const bool row_ok = r < a.rows;
    bool dead = false;                     // this warp saw a failed wait: skip work, keep barriers
    Walk wk;
    wk.init(geo);
    int i = 0;             // tiles
    int j = 0;             // pass-1 contexts ended
    int cur_ctx = -1;
    // per-context values
    int lo = 0, hi = 0, base = 0, olo = 0, ohi = 0;
    const int32_t* smap = nullptr;
    int2 pre = make_int2(0x7fffffff, 0x7fffffff);   // key positions of the coming tile
    // pass-1 state
    float m = -INFINITY, l = 0.f;
    int qpos = -1, qmin_w = 0;
    // pass-2 state
    const unsigned long long* nlse = nullptr;
    int qmin_c = 0;
    // key positions a tile needs for the causal mask (pass 1: the two
    // columns of this lane in the warp's 64; pass 2: this thread's key)
    auto load_pos = [&](int pass, int tile_key0) {
      int2 p2 = make_int2(0x7fffffff, 0x7fffffff);
      if (pass == 1) {
        const int k2 = tile_key0 + half * 64 + 2 * lane;
        if (k2 >= lo && k2 + 1 < hi) {
          p2 = *reinterpret_cast<const int2*>(smap + k2);
        } else {
          if (k2 >= lo && k2 < hi) p2.x = smap[k2];
          if (k2 + 1 >= lo && k2 + 1 < hi) p2.y = smap[k2 + 1];
        }
      } else {
        const int key = tile_key0 + quarter * 32 + lane;
        if (key >= lo && key < hi) p2.x = smap[key];
      }
      return p2;
    };
    while (wk.valid) {
      const int gi = wk.gi, b = gi / a.Hkv, g = gi % a.Hkv;
      if (!dead) dead = __any_sync(0xffffffffu, aborted(&s->abort_flag));
      if (wk.ctx != cur_ctx) {
        cur_ctx = wk.ctx;
        lo = a.attn_lo[b];
        hi = a.attn_hi[b];
        base = (lo / a.P) * a.P;
        smap = a.slot_map + ((int64_t)b * a.Hkv + g) * a.smax;
        if (wk.pass == 1) {
          m = -INFINITY;
          l = 0.f;
          qpos = row_ok ? a.q_pos[(int64_t)b * a.w + r / a.G] : 0x7fffffff;
          int mn = qpos;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
          qmin_w = mn;
        } else {
          olo = a.out_lo[b];
          ohi = a.out_hi[b];
          // wait (bounded) until every row of the group carries this call's tag
          if (e == 0) {
            const unsigned long long* rows = a.rowinfo + (int64_t)gi * kRows;
            bool ok = !dead;
            const uint64_t t0 = tc::globaltimer();
            while (ok) {
              bool mine = true;
#pragma unroll
              for (int q = 0; q < kRows / 32; ++q)
                mine = mine && (ld_acquire_u64(rows + q * 32 + lane) >> 32) == tag;
              if (__all_sync(0xffffffffu, mine)) break;
              const bool gone = __any_sync(0xffffffffu, aborted(&s->abort_flag));
              if (gone || tc::globaltimer() - t0 > limit) {
                if (lane == 0 && !gone) record_timeout(a, &s->abort_flag, kAtRows);
                ok = false;
              }
            }
          }
          named_bar(1, kEpiThreads);
          nlse = a.rowinfo + (int64_t)gi * kRows + idx * 64;
          int mn = 0x7fffffff;
          if (a.causal) {
            const int rr = idx * 64 + 2 * lane;
            const int* qrow = a.q_pos + (int64_t)b * a.w;
            mn = min(rr < a.rows ? qrow[rr / a.G] : 0x7fffffff,
                     rr + 1 < a.rows ? qrow[(rr + 1) / a.G] : 0x7fffffff);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
          }
          qmin_c = mn;
        }
        if (a.causal && !dead) pre = load_pos(wk.pass, base + wk.tile * kKeyTile);
      }
      const int tile_key0 = base + wk.tile * kKeyTile;
      const int buf = i & 1;
      const bool last_in_ctx = wk.left_in_context() == 1;
      // positions of this tile (loaded a tile ahead); start the next tile's
      const int2 pos = pre;
      if (a.causal && !dead && !last_in_ctx) pre = load_pos(wk.pass, tile_key0 + kKeyTile);
      if (!dead) {
        const bool w_ok = tc::mbar_wait(&s->acc_full[buf], (i >> 1) & 1, limit);
        if (!__all_sync(0xffffffffu, w_ok)) {
          if (lane == 0) record_timeout(a, &s->abort_flag, kAtAccFull);
          dead = true;
        }
      }
      if (wk.pass == 1) {
        const int key0 = tile_key0 + half * 64;
        if (!dead) {
          tc::tc_fence_after();
          bool fast = key0 >= lo && key0 + 64 <= hi;
          if (a.causal) {
            int mx = max(pos.x, pos.y);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            fast = fast && mx <= qmin_w;
          }
          const uint32_t tb = tmem + lane_base + buf * 256 + mb * 128 + half * 64;
          if (fast) {
            // four 16-column blocks, each loaded while the one before is reduced
            uint32_t ra[16], rb[16];
            tc::tmem_ld16_async(tb, ra);
#pragma unroll 1
            for (int blk = 0; blk < 4; blk += 2) {
              tc::tmem_wait16(ra);
              tc::tmem_ld16_async(tb + (blk + 1) * 16, rb);
              if (row_ok) p1_fast(ra, a.scale, m, l);
              tc::tmem_wait16(rb);
              if (blk == 0) {
                tc::tmem_ld16_async(tb + 32, ra);
              } else {   // every column is in registers: the buffer is free
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&s->acc_free[buf]);
              }
              if (row_ok) p1_fast(rb, a.scale, m, l);
            }
          } else {
            // range ends or causal mask inside the tile (rare): one block at a time
#pragma unroll 1
            for (int blk = 0; blk < 4; ++blk) {
              uint32_t ra[16];
              tc::tmem_ld16_async(tb + blk * 16, ra);
              tc::tmem_wait16(ra);
              if (blk == 3) {
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&s->acc_free[buf]);
              }
              p1_masked(ra, blk * 16, pos, row_ok, key0, lo, hi, a.causal, qpos, a.scale, m, l);
            }
          }
        } else {
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&s->acc_free[buf]);
        }
        if (last_in_ctx) {
          // the context's partial (max, sum) of this row and column half
          const int slot = wk.wave * (int)gridDim.x + geo.share_of(wk.wave, blockIdx.x) + gi;
          if (row_ok && !dead) a.part[((int64_t)slot * kRows + r) * 2 + half] = make_float2(m, l);
          if (j >= kRing && !dead &&
              !__all_sync(0xffffffffu,
                          tc::mbar_wait(&s->p1e[j % kRing], ((j / kRing) - 1) & 1, limit))) {
            if (lane == 0) record_timeout(a, &s->abort_flag, kAtP1e);
            dead = true;
          }
          tc::mbar_arrive(&s->p1d[j % kRing]);
          ++j;
        }
      } else {
        const int key = tile_key0 + quarter * 32 + lane;
        const int kpos = pos.x;
        float cs = 0.f;
        const uint32_t tb = tmem + lane_base + buf * 256 + idx * 64;
        if (!dead) {
          tc::tc_fence_after();
          const bool masked = a.causal && !__all_sync(0xffffffffu, kpos <= qmin_c);
          const int* qrow = a.q_pos + (int64_t)b * a.w;
          uint32_t ra[16], rb[16];
          tc::tmem_ld16_async(tb, ra);
#pragma unroll 1
          for (int blk = 0; blk < 4; blk += 2) {
            tc::tmem_wait16(ra);
            tc::tmem_ld16_async(tb + (blk + 1) * 16, rb);
            cs += p2_sum(ra, nlse + blk * 16, qrow, idx * 64 + blk * 16, a.rows, a.G, masked, kpos,
                         a.scale);
            tc::tmem_wait16(rb);
            if (blk == 0) tc::tmem_ld16_async(tb + 32, ra);
            cs += p2_sum(rb, nlse + blk * 16 + 16, qrow, idx * 64 + blk * 16 + 16, a.rows, a.G,
                         masked, kpos, a.scale);
          }
          if (idx != 0) {
            tmem_st1(tb, cs);
            tmem_wait_st();
          }
          tc::tc_fence_before();
        }
        named_bar(2 + quarter, 128);
        if (idx == 0 && !dead) {
          tc::tc_fence_after();
          const uint32_t t0 = tmem + lane_base + buf * 256;
          float p1, p2, p3;
          tmem_ld3(t0 + 64, t0 + 128, t0 + 192, p1, p2, p3);
          const float total = ((cs + p1) + p2) + p3;
          tc::tc_fence_before();
          if (key >= olo && key < ohi && key >= lo && key < hi && key < a.scores_stride) {
            float* out = a.scores + (int64_t)gi * a.scores_stride + key;
            *out = a.accumulate ? *out + total : total;
          }
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s->acc_free[buf]);
      }
      ++i;
      wk.next();
    }
  }
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
  // the last CTA to finish clears the counters for the next call
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned n = atomicAdd(a.exit_count, 1u);
    if (n == gridDim.x - 1) {
      __threadfence();
      for (int x = 0; x < a.groups; ++x) a.cnt[x] = 0u;
      *a.epoch = *a.epoch + 1u;
      *a.exit_count = 0u;
      __threadfence();
    }
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

namespace {

size_t ctrl_bytes(int groups) { return align_up(kCtrlHead + (size_t)4 * groups, 256); }

int choose_waves(int groups, int n_tiles_max) {
  // three waves of keys in L2 at a time, each at most 24 MB
  const double bytes = (double)groups * n_tiles_max * kKTileBytes;
  int W = (int)((bytes + 24.0 * (1 << 20) - 1) / (24.0 * (1 << 20)));
  return std::max(1, std::min(W, groups));
}

}  // namespace

// Largest number of tiles of one CTA's segment, from the host's bounds.
static int max_segment_tiles(int groups, int W, int n_tiles_max, int C) {
  const int wave_groups = cdiv(groups, W);
  return cdiv(wave_groups * n_tiles_max, C) + 1;
}

bool score_fused_applicable(const se_paged_kv* kv, int w, int n_max, int n_sm, int smem_optin) {
  if ((size_t)smem_optin < kSmemBytes) return false;
  const int G = kv->Hq / kv->Hkv;
  const int groups = kv->B * kv->Hkv;
  const int n_tiles_max = cdiv(n_max + kv->page_size, kKeyTile);
  if (w * G > kRows || kv->B > kMaxB || n_tiles_max < 8 || n_sm < 1 || n_sm > kMaxCTAs)
    return false;
  const int W = choose_waves(groups, n_tiles_max);
  // pass-1 contexts of two consecutive segments fit the decision ring
  return 2 * (max_segment_tiles(groups, W, n_tiles_max, n_sm) + 1) <= kRing;
}

size_t score_fused_ctrl_bytes(const se_paged_kv* kv) { return ctrl_bytes(kv->B * kv->Hkv); }

size_t score_fused_ws(const se_paged_kv* kv, int w, int n_max) {
  const int groups = kv->B * kv->Hkv;
  const int n_tiles_max = cdiv(n_max + kv->page_size, kKeyTile);
  const int W = choose_waves(groups, n_tiles_max);
  WsCarver c(nullptr);
  c.take<uint8_t>(ctrl_bytes(groups));
  c.take<unsigned long long>((size_t)groups * kRows);
  c.take<float2>(((size_t)W * kMaxCTAs + groups) * kRows * 2);
  (void)w;
  return c.bytes();
}

se_status launch_score_fused(const se_paged_kv* kv, const CUtensorMap& kmap, const CUtensorMap& qmap,
                             int w, const int32_t* q_pos, const int32_t* attn_lo,
                             const int32_t* attn_hi, const int32_t* out_lo, const int32_t* out_hi,
                             int causal, int accumulate, int n_max, float* scores,
                             int64_t scores_stride, void* ws, int n_sm, cudaStream_t st) {
  static std::atomic<uint64_t> attr{0};
  if (!allow_smem(reinterpret_cast<const void*>(&score_fused_tc), (int)kSmemBytes, attr))
    return SE_ERR_CUDA;
  const int G = kv->Hq / kv->Hkv;
  const int groups = kv->B * kv->Hkv;
  const int n_tiles_max = cdiv(n_max + kv->page_size, kKeyTile);
  FusedArgs a{};
  a.B = kv->B; a.Hq = kv->Hq; a.Hkv = kv->Hkv; a.G = G; a.w = w; a.P = kv->page_size;
  a.rows = w * G; a.groups = groups;
  a.max_pages_per_seq = kv->max_pages_per_seq;
  a.block_table = kv->block_table; a.slot_map = kv->slot_map;
  a.smax = (int64_t)kv->max_pages_per_seq * kv->page_size;
  a.q_pos = q_pos; a.attn_lo = attn_lo; a.attn_hi = attn_hi; a.out_lo = out_lo; a.out_hi = out_hi;
  a.causal = causal; a.accumulate = accumulate; a.n_max = n_max;
  a.scores = scores; a.scores_stride = scores_stride;
  uint8_t* base = static_cast<uint8_t*>(ws);
  a.limit_override = reinterpret_cast<const unsigned long long*>(base);
  a.exit_count = reinterpret_cast<unsigned int*>(base + 8);
  a.diag = reinterpret_cast<unsigned int*>(base + 12);
  a.epoch = reinterpret_cast<unsigned int*>(base + 16);
  a.cnt = reinterpret_cast<unsigned int*>(base + kCtrlHead);
  WsCarver c(ws);
  c.take<uint8_t>(ctrl_bytes(groups));
  a.rowinfo = c.take<unsigned long long>((size_t)groups * kRows);
  a.part = c.take<float2>(((size_t)choose_waves(groups, n_tiles_max) * kMaxCTAs + groups) * kRows * 2);
  a.W = choose_waves(groups, n_tiles_max);
  a.status = kv->status;
  a.scale = kLog2e / sqrtf((float)kD);

  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_sm);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, score_fused_tc, kmap, qmap, a) != cudaSuccess) return SE_ERR_CUDA;
  return SE_OK;
}

size_t score_fused_smem_bytes() { return kSmemBytes; }

}  // namespace se
