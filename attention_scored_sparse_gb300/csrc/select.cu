// Per-KV-head selection of the entries to retain.
//
// TOPK        SparseEngine "How it works" (SnapKV keeps the top entries per
//             KV head after the last prompt chunk; H2O heavy hitters; Quest
//             top pages): avg-pool over the candidate range, rank by (score
//             desc, slot asc), keep k plus a forced range.  One CTA per
//             (sequence, head): scores staged in shared memory, pooled into
//             order-preserving integer keys held in registers, a 3-pass
//             (11/11/10-bit) block radix select finds the k-th key, and two
//             block scans emit the kept slots in ascending order.
// KARA_CHUNK  KARA Method 1-2 (top-K candidates, Token2Chunk): one warp per
//             (sequence, head); candidates, chunk scores, greedy fill and
//             top-up are warp argmax rounds over registers.
// EVICT_ONE   SparseEngine "What it is" (H2O persistent scores + physical
//             eviction): one warp per (sequence, head) argmin.
#include <cooperative_groups.h>

#include "se_common.cuh"

namespace se {

struct SelectArgs {
  int B, Hkv;
  const float* scores;
  int64_t stride;
  const int32_t* cand_lo;
  const int32_t* cand_hi;
  const int32_t* force_lo;
  const int32_t* force_hi;
  int32_t* keep;
  int32_t keep_stride;
  int32_t* n_keep;
  int32_t* status;
};

template <int ITEMS>
SE_DEV int padded(int e) { return e + e / ITEMS; }

// Keys of this thread's ITEMS consecutive candidates e0 + i, i < ITEMS, from
// the scores in shared memory (element e at padded index e - xbase; n_loaded
// elements from xbase on): the sum over the pool window (neighbours outside
// [0, n) are absent), as an order-preserving uint -- the window sum ranks
// like the window mean.  Candidates at or past r_end get key 0, forced ones
// (slot in [flo, fhi)) too; returns how many were forced.  HALO >= 0: the
// window half-width at compile time, each window value read once; HALO < 0:
// the half-width pool / 2 at run time.
template <int ITEMS, int HALO>
SE_DEV int pooled_keys(const float* s_sc, int e0, int r_end, int n, int xbase, int n_loaded,
                       int pool, int lo, int flo, int fhi, bool bad, uint32_t (&key)[ITEMS]) {
  int n_forced_in = 0;
  if constexpr (HALO >= 0) {
    float w[ITEMS + 2 * HALO];
#pragma unroll
    for (int i = 0; i < ITEMS + 2 * HALO; ++i) {
      const int ee = e0 - HALO + i;
      const bool in = !bad && ee >= 0 && ee < n && ee - xbase < n_loaded;
      w[i] = in ? s_sc[padded<ITEMS>(ee - xbase)] : 0.f;
    }
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int e = e0 + i;
      key[i] = 0u;
      if (!bad && e < r_end) {
        const int slot = lo + e;
        if (slot >= flo && slot < fhi) {
          n_forced_in++;
        } else {
          float acc = 0.f;
#pragma unroll
          for (int d = 0; d <= 2 * HALO; ++d) acc += w[i + d];
          key[i] = float_key(acc);
        }
      }
    }
  } else {
    const int halo = pool / 2;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int e = e0 + i;
      key[i] = 0u;
      if (!bad && e < r_end) {
        const int slot = lo + e;
        if (slot >= flo && slot < fhi) {
          n_forced_in++;
        } else {
          float v;
          if (pool > 1) {
            v = 0.f;
            for (int d = -halo; d <= halo; ++d) {
              const int ee = e + d;
              if (ee >= 0 && ee < n) v += s_sc[padded<ITEMS>(ee - xbase)];
            }
          } else {
            v = s_sc[padded<ITEMS>(e - xbase)];
          }
          key[i] = float_key(v);
        }
      }
    }
  }
  return n_forced_in;
}

// grid: (Hkv, B), 1024 threads, dynamic smem (1024*(ITEMS+1)+64) floats.
template <int ITEMS>
__global__ void __launch_bounds__(1024, 1) topk_kernel(SelectArgs a, int pool, int k) {
  pdl_enter();
  extern __shared__ float s_sc[];
  __shared__ int tmp[33];
  __shared__ int hist[2048];
  __shared__ int s_digit, s_rem;
  __shared__ int s_before_force;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int lo = a.cand_lo[b], hi = a.cand_hi[b];
  const int flo = a.force_lo ? a.force_lo[b] : 0;
  const int fhi = a.force_hi ? a.force_hi[b] : 0;
  const int n = hi - lo;
  const int nf = max(fhi - flo, 0);
  if (n < 0 || n > 1024 * ITEMS) {
    if (tid == 0) set_status(a.status, SE_ERR_BOUNDS);
    return;
  }
  const float* row = a.scores + ((int64_t)b * a.Hkv + h) * a.stride;
  {
    // every load of the thread in flight before the first store
    float v[ITEMS];
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) v[i] = tid + i * 1024 < n ? row[lo + tid + i * 1024] : 0.f;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i)
      if (tid + i * 1024 < n) s_sc[padded<ITEMS>(tid + i * 1024)] = v[i];
  }
  if (tid == 0) s_before_force = 0;
  __syncthreads();

  uint32_t key[ITEMS];
  const int n_forced_in =
      pooled_keys<ITEMS, -1>(s_sc, tid * ITEMS, n, n, 0, n, pool, lo, flo, fhi, false, key);
  int forced_in_total;
  block_exclusive_scan(n_forced_in, tmp, &forced_in_total);
  const int ncand = n - forced_in_total;
  const int kk = min(max(k, 0), ncand);

  // Up to 3 rounds of radix select (digits of 11, 11 and 10 bits, top first)
  // for the kk-th largest key; a round whose threshold digit keeps every key
  // under the prefix ends the search.  Wide digits spread scores that share
  // an exponent.
  uint32_t prefix = 0, pmask = 0;
  int remaining = kk;
  if (kk > 0) {
#pragma unroll 1
    for (int round = 0; round < 3; ++round) {
      const int shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
      const int nbins = round == 2 ? 1024 : 2048;
      const uint32_t dmask = (uint32_t)nbins - 1u;
      for (int i = tid; i < nbins; i += 1024) hist[i] = 0;
      __syncthreads();
      hist_add_keys<ITEMS>(hist, key, shift, dmask, pmask, prefix);
      __syncthreads();
      radix_find_digit(hist, nbins, remaining, tmp, &s_digit, &s_rem);
      prefix |= (uint32_t)s_digit << shift;
      remaining = s_rem;
      pmask |= dmask << shift;
      // every key under this prefix is kept: its lower digits decide nothing
      const bool whole_bin = hist[s_digit] == s_rem;
      __syncthreads();
      if (whole_bin) break;
    }
  }
  // keys are compared on the digits resolved so far
  const uint32_t T = kk > 0 ? prefix : 0xffffffffu;
  const uint32_t TM = kk > 0 ? pmask : 0xffffffffu;
  const int need_eq = kk > 0 ? remaining : 0;

  int c_eq = 0;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) c_eq += (key[i] != 0u && (key[i] & TM) == T) ? 1 : 0;
  int dummy;
  int eq_rank = block_exclusive_scan(c_eq, tmp, &dummy);
  bool sel[ITEMS];
  int c_sel = 0, c_sel_before_force = 0;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    sel[i] = false;
    if (key[i] != 0u) {
      if ((key[i] & TM) > T) {
        sel[i] = true;
      } else if ((key[i] & TM) == T) {
        sel[i] = eq_rank < need_eq;
        eq_rank++;
      }
    }
    c_sel += sel[i];
    c_sel_before_force += (sel[i] && lo + tid * ITEMS + i < flo) ? 1 : 0;
  }
  int total_sel;
  int pos = block_exclusive_scan(c_sel, tmp, &total_sel);
  if (total_sel + nf > a.keep_stride) {  // output row too short: report, write nothing
    if (tid == 0) set_status(a.status, SE_ERR_BOUNDS);
    return;
  }
  if (c_sel_before_force) atomicAdd(&s_before_force, c_sel_before_force);
  __syncthreads();
  const int before_force = s_before_force;
  int32_t* out = a.keep + ((int64_t)b * a.Hkv + h) * a.keep_stride;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    if (sel[i]) {
      const int slot = lo + tid * ITEMS + i;
      out[pos + (slot >= fhi && nf > 0 ? nf : 0)] = slot;
      pos++;
    }
  }
  for (int f = tid; f < nf; f += 1024) out[before_force + f] = flo + f;
  for (int p = total_sel + nf + tid; p < a.keep_stride; p += 1024) out[p] = -1;
  if (h == 0 && tid == 0 && a.n_keep) a.n_keep[b] = total_sel + nf;
}

// --------------------------------------------------------------------------
// Same selection split over a cluster of 4 CTAs per (sequence, head): CTA
// rank r owns a quarter of the candidate range (plus a pooling halo), keeps
// its keys in registers, and the cluster combines radix histograms, equal-key
// ranks and output offsets through distributed shared memory.  Four times the
// SMs of the one-CTA kernel for the few-instance, long-range case.
// grid: (4 * Hkv, B), cluster (4, 1, 1), 1024 threads.
// --------------------------------------------------------------------------
constexpr int kClusterCTAs = 4;

template <int ITEMS, int HALO>
__global__ void __cluster_dims__(kClusterCTAs, 1, 1) __launch_bounds__(1024, 1)
topk_cluster_kernel(SelectArgs a, int pool, int k) {
  pdl_enter();
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ float s_sc[];
  __shared__ int tmp[33];
  __shared__ int hist[2][2048];   // double-buffered: peers read round r while round r+1 fills the other
  __shared__ int tot[2048];       // this round's histogram summed over the cluster
  __shared__ int s_cnt[4];        // forced-in-range, equal-to-T, selected, selected-before-force
  __shared__ int s_digit, s_rem;
  const int rank = (int)cluster.block_rank();
  const int h = blockIdx.x / kClusterCTAs, b = blockIdx.y, tid = threadIdx.x;
  const int lo = a.cand_lo[b], hi = a.cand_hi[b];
  const int flo = a.force_lo ? a.force_lo[b] : 0;
  const int fhi = a.force_hi ? a.force_hi[b] : 0;
  const int n = hi - lo;
  const int nf = max(fhi - flo, 0);
  const int per = cdiv(max(n, 1), kClusterCTAs);
  const bool bad = n < 0 || per > 1024 * ITEMS;    // same for the whole cluster
  const int r0 = min(rank * per, max(n, 0)), r1 = min(r0 + per, max(n, 0));
  const int halo = pool / 2;
  const float* row = a.scores + ((int64_t)b * a.Hkv + h) * a.stride;
  // local smem index x <-> element r0 - halo + x
  const int x1 = bad ? 0 : (r1 + halo) - (r0 - halo);
  // every load of the thread in flight before the first store; the range
  // (at most 1024 ITEMS) and its two halos take at most ITEMS + 1 rounds
  // when the halos add up to 1024 or less
  if (2 * halo <= 1024) {
    float v[ITEMS + 1];
#pragma unroll
    for (int i = 0; i <= ITEMS; ++i) {
      const int x = tid + i * 1024, e = r0 - halo + x;
      v[i] = (x < x1 && e >= 0 && e < n) ? row[lo + e] : 0.f;
    }
#pragma unroll
    for (int i = 0; i <= ITEMS; ++i)
      if (tid + i * 1024 < x1) s_sc[padded<ITEMS>(tid + i * 1024)] = v[i];
  } else {
    for (int x = tid; x < x1; x += 1024) {
      const int e = r0 - halo + x;
      s_sc[padded<ITEMS>(x)] = (e >= 0 && e < n) ? row[lo + e] : 0.f;
    }
  }
  if (tid < 4) s_cnt[tid] = 0;
  __syncthreads();

  uint32_t key[ITEMS];
  const int n_forced_in = pooled_keys<ITEMS, HALO>(s_sc, r0 + tid * ITEMS, r1, n, r0 - halo, x1,
                                                   pool, lo, flo, fhi, bad, key);
  if (n_forced_in) atomicAdd(&s_cnt[0], n_forced_in);

  // Up to three radix rounds; the forced-in counts travel with round 0's
  // barrier (the histogram does not depend on k).
  uint32_t prefix = 0, pmask = 0;
  int kk = 0, remaining = 0, bin_total = 0;
#pragma unroll 1
  for (int round = 0; round < 3; ++round) {
    const int shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
    const int nbins = round == 2 ? 1024 : 2048;
    const uint32_t dmask = (uint32_t)nbins - 1u;
    // buffer round & 1 was last read by peers two rounds ago; every peer
    // has passed the previous round's cluster barrier since, after its reads
    int* hb = hist[round & 1];
    for (int i = tid; i < nbins; i += 1024) hb[i] = 0;
    __syncthreads();
    hist_add_keys<ITEMS>(hb, key, shift, dmask, pmask, prefix);
    cluster.sync();                    // every CTA's histogram (and round 0: count) is complete
    if (round == 0) {
      int forced_in_total = 0;
      for (int r = 0; r < kClusterCTAs; ++r) forced_in_total += *cluster.map_shared_rank(&s_cnt[0], r);
      kk = bad ? 0 : min(max(k, 0), n - forced_in_total);
      remaining = kk;
      if (kk == 0) break;              // same in every CTA
    }
    // each thread sums up to two bins over the cluster
    for (int j = 0; j < 2; ++j) {
      const int bin = tid + j * 1024;
      if (bin < nbins) {
        int sum = 0;
        for (int r = 0; r < kClusterCTAs; ++r) sum += *cluster.map_shared_rank(&hb[bin], r);
        tot[bin] = sum;
      }
    }
    __syncthreads();
    radix_find_digit(tot, nbins, remaining, tmp, &s_digit, &s_rem);
    prefix |= (uint32_t)s_digit << shift;
    remaining = s_rem;
    pmask |= dmask << shift;
    bin_total = tot[s_digit];
    __syncthreads();
    // every key under this prefix is kept: its lower digits decide nothing
    // (tot is the same in every CTA of the cluster, so is the decision)
    if (bin_total == remaining) break;
  }
  // keys are compared on the digits resolved so far
  const uint32_t T = kk > 0 ? prefix : 0xffffffffu;
  const uint32_t TM = kk > 0 ? pmask : 0xffffffffu;
  const int need_eq = kk > 0 ? remaining : 0;

  // keys equal to T on those digits: all of them are taken unless ties at
  // the full key cut the threshold bin; only then do they need their
  // cluster-wide rank in element order
  const bool all_eq = kk == 0 || bin_total == need_eq;
  int eq_rank = 0;
  if (!all_eq) {
    int c_eq = 0;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) c_eq += (key[i] != 0u && (key[i] & TM) == T) ? 1 : 0;
    int my_eq_total;
    eq_rank = block_exclusive_scan(c_eq, tmp, &my_eq_total);
    if (tid == 0) s_cnt[1] = my_eq_total;
    cluster.sync();
    for (int r = 0; r < rank; ++r) eq_rank += *cluster.map_shared_rank(&s_cnt[1], r);
  }
  bool sel[ITEMS];
  int c_sel = 0, c_sel_before_force = 0;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    sel[i] = false;
    if (key[i] != 0u) {
      if ((key[i] & TM) > T) {
        sel[i] = true;
      } else if ((key[i] & TM) == T) {
        sel[i] = all_eq || eq_rank < need_eq;
        eq_rank++;
      }
    }
    c_sel += sel[i];
    c_sel_before_force += (sel[i] && lo + r0 + tid * ITEMS + i < flo) ? 1 : 0;
  }
  int my_sel_total;
  int pos = block_exclusive_scan(c_sel, tmp, &my_sel_total);
  if (c_sel_before_force) atomicAdd(&s_cnt[3], c_sel_before_force);
  if (tid == 0) s_cnt[2] = my_sel_total;
  cluster.sync();
  int total_sel = 0, before_force = 0;
  for (int r = 0; r < kClusterCTAs; ++r) {
    const int cs = *cluster.map_shared_rank(&s_cnt[2], r);
    if (r < rank) pos += cs;
    total_sel += cs;
    before_force += *cluster.map_shared_rank(&s_cnt[3], r);
  }
  // peers may still read this CTA's counters: arrive now, wait before leaving
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  const bool fail = bad || total_sel + nf > a.keep_stride;   // same in every CTA
  if (fail) {
    if (rank == 0 && tid == 0) set_status(a.status, SE_ERR_BOUNDS);
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
    return;
  }
  int32_t* out = a.keep + ((int64_t)b * a.Hkv + h) * a.keep_stride;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    if (sel[i]) {
      const int slot = lo + r0 + tid * ITEMS + i;
      out[pos + (slot >= fhi && nf > 0 ? nf : 0)] = slot;
      pos++;
    }
  }
  if (rank == 0) {
    for (int f = tid; f < nf; f += 1024) out[before_force + f] = flo + f;
    for (int p = total_sel + nf + tid; p < a.keep_stride; p += 1024) out[p] = -1;
    if (h == 0 && tid == 0 && a.n_keep) a.n_keep[b] = total_sel + nf;
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// --------------------------------------------------------------------------
// Kara Token2Chunk: one warp per (b, h); compressible window <= 32*IT slots.
// --------------------------------------------------------------------------

struct ArgBest {
  float s;
  int idx;  // element index (tie: smaller wins)
};

SE_DEV ArgBest warp_argmax(ArgBest v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ArgBest w;
    w.s = __shfl_xor_sync(0xffffffffu, v.s, o);
    w.idx = __shfl_xor_sync(0xffffffffu, v.idx, o);
    if (w.s > v.s || (w.s == v.s && w.idx < v.idx)) v = w;
  }
  return v;
}

// j-th set bit (0-based) of a little-endian multi-word mask, -1 if none.
template <int IT>
SE_DEV int select_bit(const uint32_t* words, int j) {
#pragma unroll
  for (int w = 0; w < IT; ++w) {
    const int c = __popc(words[w]);
    if (j < c) {
      uint32_t x = words[w];
      for (int t = 0; t < j; ++t) x &= x - 1;
      return w * 32 + (__ffs(x) - 1);
    }
    j -= c;
  }
  return -1;
}

template <int IT>
__global__ void __launch_bounds__(256) kara_chunk_kernel(SelectArgs a, int n_cand, int budget,
                                                         float coef) {
  pdl_enter();
  __shared__ float s_sc[8][32 * IT];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int inst = blockIdx.x * 8 + warp;
  if (inst >= a.B * a.Hkv) return;
  const int b = inst / a.Hkv, h = inst % a.Hkv;
  const int lo = a.cand_lo[b], hi = a.cand_hi[b];
  const int flo = a.force_lo ? a.force_lo[b] : 0;
  const int fhi = a.force_hi ? a.force_hi[b] : 0;
  const int nf = max(fhi - flo, 0);
  const int n = hi - lo;
  if (n < 0 || n > 32 * IT || n_cand > 32) {
    if (lane == 0) set_status(a.status, SE_ERR_BOUNDS);
    return;
  }
  const float* row = a.scores + ((int64_t)b * a.Hkv + h) * a.stride;
  float* sc = s_sc[warp];
  float s[IT];
  bool cand_ok[IT], is_c[IT], ret[IT];
#pragma unroll
  for (int i = 0; i < IT; ++i) {
    const int e = i * 32 + lane;
    const int slot = lo + e;
    const bool inr = e < n && !(slot >= flo && slot < fhi);
    s[i] = e < n ? row[lo + e] : 0.f;
    if (e < 32 * IT) sc[e] = s[i];
    cand_ok[i] = inr;
    is_c[i] = false;
    ret[i] = false;
  }
  __syncwarp();
  int n_avail = 0;
#pragma unroll
  for (int i = 0; i < IT; ++i) n_avail += __popc(__ballot_sync(0xffffffffu, cand_ok[i]));
  const int kc = min(n_cand, n_avail);
  const int bud = min(budget, n_avail);
  // 1) top-kc discrete candidates by (score desc, index asc)
  for (int r = 0; r < kc; ++r) {
    ArgBest v{-INFINITY, 0x7fffffff};
#pragma unroll
    for (int i = 0; i < IT; ++i) {
      const int e = i * 32 + lane;
      if (cand_ok[i] && !is_c[i] && (s[i] > v.s || (s[i] == v.s && e < v.idx))) v = ArgBest{s[i], e};
    }
    v = warp_argmax(v);
    if ((v.idx & 31) == lane) {
#pragma unroll
      for (int i = 0; i < IT; ++i)
        if (i == (v.idx >> 5)) is_c[i] = true;
    }
  }
  uint32_t words[IT];
#pragma unroll
  for (int i = 0; i < IT; ++i) {
    words[i] = __ballot_sync(0xffffffffu, is_c[i]);
    ret[i] = is_c[i];
  }
  int count = kc;
  // 2) chunk between consecutive candidates j, j+1 (lane j)
  const int n_chunks = max(kc - 1, 0);
  float csc = -INFINITY;
  int ca = 0, cb = 0;
  if (lane < n_chunks) {
    ca = select_bit<IT>(words, lane);
    cb = select_bit<IT>(words, lane + 1);
    csc = (sc[ca] + sc[cb]) * 0.5f - coef * (float)(cb - ca);
  }
  bool visited = lane >= n_chunks;
  for (int r = 0; r < n_chunks; ++r) {
    ArgBest v{-INFINITY, 0x7fffffff};
    if (!visited) v = ArgBest{csc, ca};
    v = warp_argmax(v);
    // the winner is the chunk starting at v.idx
    const bool win = !visited && ca == v.idx;
    const unsigned wm = __ballot_sync(0xffffffffu, win);
    const int wl = __ffs(wm) - 1;
    const int a0 = __shfl_sync(0xffffffffu, ca, wl);
    const int b0 = __shfl_sync(0xffffffffu, cb, wl);
    if (lane == wl) visited = true;
    const int interior = b0 - a0 - 1;
    if (interior > 0 && count + interior <= bud) {
      count += interior;
#pragma unroll
      for (int i = 0; i < IT; ++i) {
        const int e = i * 32 + lane;
        if (e > a0 && e < b0) ret[i] = true;
      }
    }
  }
  // 3) top up with the best remaining single tokens
  while (count < bud) {
    ArgBest v{-INFINITY, 0x7fffffff};
#pragma unroll
    for (int i = 0; i < IT; ++i) {
      const int e = i * 32 + lane;
      if (cand_ok[i] && !ret[i] && (s[i] > v.s || (s[i] == v.s && e < v.idx))) v = ArgBest{s[i], e};
    }
    v = warp_argmax(v);
    if ((v.idx & 31) == lane) {
#pragma unroll
      for (int i = 0; i < IT; ++i)
        if (i == (v.idx >> 5)) ret[i] = true;
    }
    count++;
  }
  // 4) emit retained slots ascending, forced range in slot order
  if (count + nf > a.keep_stride) {
    if (lane == 0) set_status(a.status, SE_ERR_BOUNDS);
    return;
  }
  int32_t* out = a.keep + ((int64_t)b * a.Hkv + h) * a.keep_stride;
  int before_force = 0;
#pragma unroll
  for (int i = 0; i < IT; ++i) {
    const uint32_t m = __ballot_sync(0xffffffffu, ret[i] && lo + i * 32 + lane < flo);
    before_force += __popc(m);
  }
  int base = 0;
#pragma unroll
  for (int i = 0; i < IT; ++i) {
    const uint32_t m = __ballot_sync(0xffffffffu, ret[i]);
    if (ret[i]) {
      const int slot = lo + i * 32 + lane;
      const int p = base + __popc(m & ((1u << lane) - 1u));
      out[p + (slot >= fhi && nf > 0 ? nf : 0)] = slot;
    }
    base += __popc(m);
  }
  for (int f = lane; f < nf; f += 32) out[before_force + f] = flo + f;
  if (h == 0 && lane == 0 && a.n_keep) a.n_keep[b] = count + nf;
}

// --------------------------------------------------------------------------
// H2O evict-one: one warp per (b, h).
// --------------------------------------------------------------------------
// (v, pos) ranks below (bv, bpos): lower running score, ties to the higher
// position (the mirror of the selection tie rule).
SE_DEV bool evict_before(float v, int pos, float bv, int bpos, int bslot) {
  return bslot < 0 || v < bv || (v == bv && pos > bpos);
}

// grid: B * Hkv, 128 threads (one CTA per (sequence, head)).  Each thread
// scans every 128th slot with four loads in flight, then warp shuffles and
// shared memory pick the minimum.
__global__ void __launch_bounds__(128) evict_one_kernel(SelectArgs a, const int32_t* ctx_len,
                                                        const int32_t* logical_len,
                                                        const int32_t* slot_map, int64_t smax,
                                                        int budget, int recent) {
  pdl_enter();
  __shared__ float s_v[4];
  __shared__ int s_p[4], s_s[4];
  const int inst = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = inst / a.Hkv, h = inst % a.Hkv;
  const int ctx = ctx_len[b];
  int32_t* out = a.keep + (int64_t)b * a.Hkv + h;
  if (ctx <= budget) {
    if (tid == 0) *out = -1;
    return;
  }
  const int recent_from = logical_len[b] - recent;
  const float* acc = a.scores + ((int64_t)b * a.Hkv + h) * a.stride;
  const int32_t* sm = slot_map + ((int64_t)b * a.Hkv + h) * smax;
  float best = INFINITY;
  int bpos = -1, bslot = -1;
  for (int s0 = tid; s0 < ctx; s0 += 4 * 128) {
    int pos[4];
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int sl = s0 + u * 128;
      pos[u] = sl < ctx ? sm[sl] : INT_MAX;
      v[u] = sl < ctx ? acc[sl] : 0.f;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (pos[u] < recent_from && evict_before(v[u], pos[u], best, bpos, bslot)) {
        best = v[u];
        bpos = pos[u];
        bslot = s0 + u * 128;
      }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v = __shfl_xor_sync(0xffffffffu, best, o);
    const int p = __shfl_xor_sync(0xffffffffu, bpos, o);
    const int sl = __shfl_xor_sync(0xffffffffu, bslot, o);
    if (sl >= 0 && evict_before(v, p, best, bpos, bslot)) { best = v; bpos = p; bslot = sl; }
  }
  if (lane == 0) { s_v[warp] = best; s_p[warp] = bpos; s_s[warp] = bslot; }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < 4; ++w)
      if (s_s[w] >= 0 && evict_before(s_v[w], s_p[w], best, bpos, bslot)) {
        best = s_v[w]; bpos = s_p[w]; bslot = s_s[w];
      }
    *out = bslot;
  }
}

template <int ITEMS>
static se_status launch_topk_t(const SelectArgs& a, int pool, int k, cudaStream_t st) {
  const size_t smem = (size_t)(1024 * (ITEMS + 1) + 64) * sizeof(float);
  static std::atomic<uint64_t> attr{0};
  if (!allow_smem(reinterpret_cast<const void*>(&topk_kernel<ITEMS>), (int)smem, attr))
    return SE_ERR_CUDA;
  se_launch(topk_kernel<ITEMS>, dim3(a.Hkv, a.B), 1024, smem, st, a, pool, k);
  return SE_OK;
}

template <int ITEMS, int HALO>
static se_status launch_topk_cluster_h(const SelectArgs& a, int pool, int k, cudaStream_t st) {
  const size_t smem = (size_t)(1024 * (ITEMS + 1) + 64) * sizeof(float);
  static std::atomic<uint64_t> attr{0};
  if (!allow_smem(reinterpret_cast<const void*>(&topk_cluster_kernel<ITEMS, HALO>), (int)smem, attr))
    return SE_ERR_CUDA;
  se_launch(topk_cluster_kernel<ITEMS, HALO>, dim3(kClusterCTAs * a.Hkv, a.B), 1024, smem, st, a,
            pool, k);
  return SE_OK;
}

// the SnapKV pooling width (7) with its window unrolled; any other width at run time
template <int ITEMS>
static se_status launch_topk_cluster_t(const SelectArgs& a, int pool, int k, cudaStream_t st) {
  if (pool == 7) return launch_topk_cluster_h<ITEMS, 3>(a, pool, k, st);
  return launch_topk_cluster_h<ITEMS, -1>(a, pool, k, st);
}

se_status launch_topk(const SelectArgs& a, int pool, int k, int n_max, cudaStream_t st) {
  // long candidate ranges: four CTAs per (sequence, head) in a cluster
  if (n_max > 8192) {
    const int items = cdiv(cdiv(n_max, kClusterCTAs) + 8, 1024);
    if (items <= 2) return launch_topk_cluster_t<2>(a, pool, k, st);
    if (items <= 4) return launch_topk_cluster_t<4>(a, pool, k, st);
    if (items <= 8) return launch_topk_cluster_t<8>(a, pool, k, st);
    if (items <= 16) return launch_topk_cluster_t<16>(a, pool, k, st);
    if (items <= 32) return launch_topk_cluster_t<32>(a, pool, k, st);
    if (items <= 48) return launch_topk_cluster_t<48>(a, pool, k, st);
    return SE_ERR_UNSUPPORTED;
  }
  const int items = cdiv(max(n_max, 1), 1024);
  if (items <= 1) return launch_topk_t<1>(a, pool, k, st);
  if (items <= 2) return launch_topk_t<2>(a, pool, k, st);
  if (items <= 4) return launch_topk_t<4>(a, pool, k, st);
  if (items <= 8) return launch_topk_t<8>(a, pool, k, st);
  if (items <= 16) return launch_topk_t<16>(a, pool, k, st);
  if (items <= 32) return launch_topk_t<32>(a, pool, k, st);
  if (items <= 48) return launch_topk_t<48>(a, pool, k, st);
  return SE_ERR_UNSUPPORTED;
}

se_status launch_topk_select_pages(int B, int Hkv, const float* U, int64_t stride,
                                   const int32_t* cand_lo, const int32_t* cand_hi,
                                   const int32_t* force_lo, const int32_t* force_hi, int32_t* out,
                                   int32_t out_stride, int32_t* n_sel, int32_t* status, int top,
                                   int n_max, cudaStream_t st) {
  SelectArgs a{B, Hkv, U, stride, cand_lo, cand_hi, force_lo, force_hi, out, out_stride, n_sel,
               status};
  return launch_topk(a, 1, top, n_max, st);
}

}  // namespace se

using namespace se;

extern "C" se_status se_topk_select(const se_paged_kv* kv, const float* scores,
                                    int64_t scores_stride, const se_select_params* params,
                                    const int32_t* cand_lo, const int32_t* cand_hi,
                                    const int32_t* force_lo, const int32_t* force_hi,
                                    int32_t* keep_idx, int32_t keep_stride, int32_t* n_keep,
                                    void* stream) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (params == nullptr || scores == nullptr || keep_idx == nullptr) return SE_ERR_INVALID_ARG;
  if ((force_lo == nullptr) != (force_hi == nullptr)) return SE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SelectArgs a{kv->B, kv->Hkv, scores, scores_stride, cand_lo, cand_hi, force_lo, force_hi,
               keep_idx, keep_stride, n_keep, kv->status};
  const se_select_params& p = *params;
  if (p.mode == SE_SELECT_TOPK) {
    if (cand_lo == nullptr || cand_hi == nullptr || p.pool_kernel < 1 || p.pool_kernel % 2 == 0 ||
        p.k < 0 || p.n_max < 0)
      return SE_ERR_INVALID_ARG;
    s = launch_topk(a, p.pool_kernel, p.k, p.n_max, st);
    if (s != SE_OK) return s;
    return se_last_launch_status();
  }
  if (p.mode == SE_SELECT_KARA_CHUNK) {
    if (cand_lo == nullptr || cand_hi == nullptr || p.k < 1 || p.k > 32 || p.chunk_budget < 0 ||
        p.n_max < 0)
      return SE_ERR_INVALID_ARG;
    const int blocks = cdiv(kv->B * kv->Hkv, 8);
    if (p.n_max <= 256) {
      se_launch(kara_chunk_kernel<8>, blocks, 256, 0, st, a, p.k, p.chunk_budget, p.chunk_coef);
    } else if (p.n_max <= 512) {
      se_launch(kara_chunk_kernel<16>, blocks, 256, 0, st, a, p.k, p.chunk_budget, p.chunk_coef);
    } else {
      return SE_ERR_UNSUPPORTED;
    }
    return se_last_launch_status();
  }
  if (p.mode == SE_SELECT_EVICT_ONE) {
    if (p.budget < 0 || p.recent < 0) return SE_ERR_INVALID_ARG;
    se_launch(evict_one_kernel, kv->B * kv->Hkv, 128, 0, st, a, kv->ctx_len, kv->logical_len, kv->slot_map,
                                             (int64_t)kv->max_pages_per_seq * kv->page_size,
                                             p.budget, p.recent);
    return se_last_launch_status();
  }
  return SE_ERR_INVALID_ARG;
}
