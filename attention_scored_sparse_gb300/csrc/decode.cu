// Decode attention over a view of the paged cache.
//
// SparseEngine "How it works" (AttentionView): View = BuildView(C, I),
// o = Attention(q, View) -- the view is every resident entry, the resident
// slots of a list of blocks (Quest pages) or a list of slots.
//
// Bandwidth-bound design (each K/V byte is used by the G query heads of its
// group and nothing else): split-K over the view (ranges of entries, one
// CTA each, four CTAs per SM; see the work split below), a half-warp per
// group of 16/G entries with 16-byte row loads (a 256-byte bf16 row is one
// coalesced half-warp load), the group's G queries pre-scaled by
// log2(e)/sqrt(D) in registers, an xor reduce-scatter of the partial dot
// products, one exponential per (entry, head) and a base-2 online softmax.
// Half-warp states merge in shared memory into one partial per segment; the
// last CTA to finish a segment of a (sequence, KV group) merges the partials
// and, for H2O, adds sum_h p_{h,j} to the running scores from the logits the
// CTAs stored.
#include <algorithm>

#include <cooperative_groups.h>

#include "compact_ws.cuh"
#include "tc_primitives.cuh"

namespace se {

namespace cg = cooperative_groups;

template <typename T, int V>
SE_DEV void load_row(const T* p, float* f) {
  if constexpr (sizeof(T) == 2 && V == 8) {
    unpack8_bf16(ldg_nc_v4(p), f);
  } else if constexpr (sizeof(T) == 2 && V == 4) {
    uint2 u;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(u.x), "=r"(u.y) : "l"(p));
    f[0] = bf16lo(u.x); f[1] = bf16hi(u.x); f[2] = bf16lo(u.y); f[3] = bf16hi(u.y);
  } else if constexpr (sizeof(T) == 4 && V == 4) {
    const uint4 u = ldg_nc_v4(p);
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
  } else {
    static_assert(sizeof(T) == 4 && V == 8, "row layout");
    const uint4 u = ldg_nc_v4(p);
    const uint4 w = ldg_nc_v4(p + 4);
    f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
    f[4] = __uint_as_float(w.x); f[5] = __uint_as_float(w.y);
    f[6] = __uint_as_float(w.z); f[7] = __uint_as_float(w.w);
  }
}

SE_DEV float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Work split.  The view entries of every (b, g) unit are padded to sp
// slices of SE = 128 / G entries (one iteration of the 8 half-warps); the
// ts = units x sp slices, in unit order, are cut into n_cta ranges, one per
// CTA, in one of two ways:
//   aligned (k_al > 0): each unit in k_al chunks of w_al slices (the last
//     one shorter); a range never crosses a unit;
//   stream (k_al == 0, "stream-K"): n_cta contiguous ranges of nearly equal
//     length over all slices; a range that crosses a unit boundary makes one
//     segment per unit.  Equal ranges keep every CTA busy to the end when
//     the aligned chunks would leave a ragged last wave.
// Every segment leaves a partial (m, l, o) that the last CTA to finish a
// segment of the unit merges.
struct DecodeArgs {
  se_paged_kv kv;
  const void* q;
  int view;
  const int32_t* sel;
  int32_t sel_stride;
  int32_t n_sel;
  int sp;          // slices per unit
  int64_t ts;      // slices in all = units * sp
  int n_cta;       // CTAs (ranges), 1 <= n_cta <= ts
  int k_al;        // aligned split: chunks per unit, 0 for the stream split
  int w_al;        // aligned split: slices per chunk
  int max_parts;   // partial slots per unit
  float* part;     // [units][max_parts][G][D + 2]
  float* logits;   // [B][Hkv][max_entries][G] or null
  int max_entries;
  void* out;          // o [B][Hq][D]
  float* acc;         // H2O running scores or null
  int64_t acc_stride;
  int32_t* done;      // [units] segments finished (zero at the launch; the last CTA of a unit resets it)
  int k_cl;           // cluster split: CTAs per unit (one cluster each); 0 for the kernels above
};

// Slices [start, end) of CTA c's range.
SE_HD int64_t range_start(const DecodeArgs& a, int c) {
  if (a.k_al > 0) {
    const int64_t off = (int64_t)(c % a.k_al) * a.w_al;
    return (int64_t)(c / a.k_al) * a.sp + (off < a.sp ? off : a.sp);
  }
  return (int64_t)c * a.ts / a.n_cta;
}
SE_HD int64_t range_end(const DecodeArgs& a, int c) {
  if (a.k_al > 0) {
    const int64_t off = (int64_t)(c % a.k_al + 1) * a.w_al;
    return (int64_t)(c / a.k_al) * a.sp + (off < a.sp ? off : a.sp);
  }
  return (int64_t)(c + 1) * a.ts / a.n_cta;
}
// CTA whose stream range holds slice x.
SE_HD int stream_owner(const DecodeArgs& a, int64_t x) {
  return (int)(((x + 1) * a.n_cta - 1) / a.ts);
}
// The CTAs with a segment of unit u: first and count.
SE_HD void unit_parts(const DecodeArgs& a, int u, int* first, int* n) {
  if (a.k_al > 0) {
    *first = u * a.k_al;
    *n = a.k_al;
    return;
  }
  const int64_t u0 = (int64_t)u * a.sp;
  *first = stream_owner(a, u0);
  *n = stream_owner(a, u0 + a.sp - 1) - *first + 1;
}

// Resident slot of view entry e of (b, g), or -1.
SE_DEV int view_slot(const DecodeArgs& a, int b, int g, int e, int ctx) {
  if (a.view == SE_VIEW_DENSE) return e < ctx ? e : -1;
  const int32_t* sel = a.sel + ((int64_t)b * a.kv.Hkv + g) * a.sel_stride;
  if (a.view == SE_VIEW_PAGES) {
    const int P = a.kv.page_size;
    const int i = e / P;
    if (i >= a.n_sel) return -1;
    const int blk = sel[i];
    const int s = blk * P + e % P;
    return (blk >= 0 && s < ctx) ? s : -1;
  }
  if (e >= a.n_sel) return -1;
  const int s = sel[e];
  return (s >= 0 && s < ctx) ? s : -1;
}

SE_DEV int view_entries(const DecodeArgs& a, int ctx) {
  if (a.view == SE_VIEW_DENSE) return ctx;
  if (a.view == SE_VIEW_PAGES) return a.n_sel * a.kv.page_size;
  return a.n_sel;
}

// The G logits of one entry (G consecutive floats, 4 G-byte aligned: the
// logits array is 256-byte aligned and holds G floats per entry) through
// L2, as 16-, 8- or 4-byte loads; zeros when !ok.
template <int G>
SE_DEV void load_logits(const float* p, bool ok, float (&v)[G]) {
  if constexpr (G % 4 == 0) {
#pragma unroll
    for (int j = 0; j < G; j += 4) {
      const float4 f = ok ? __ldcg(reinterpret_cast<const float4*>(p + j)) : make_float4(0.f, 0.f, 0.f, 0.f);
      v[j] = f.x; v[j + 1] = f.y; v[j + 2] = f.z; v[j + 3] = f.w;
    }
  } else if constexpr (G == 2) {
    const float2 f = ok ? __ldcg(reinterpret_cast<const float2*>(p)) : make_float2(0.f, 0.f);
    v[0] = f.x; v[1] = f.y;
  } else {
#pragma unroll
    for (int j = 0; j < G; ++j) v[j] = ok ? __ldcg(p + j) : 0.f;
  }
}

// Merges the n_parts partials of unit u = (b, g), writes o and updates the
// running scores.  Run by the last CTA to finish a segment of u (128 threads).
template <typename T, int D, int G>
SE_DEV void merge_chunks(const DecodeArgs& a, int u, int n_parts) {
  __shared__ float s_M[G], s_invL[G];
  T* out = static_cast<T*>(a.out);
  float* acc = a.acc;
  const int64_t acc_stride = a.acc_stride;
  const se_paged_kv& kv = a.kv;
  const int b = u / kv.Hkv, g = u % kv.Hkv;
  const float* part = a.part + (int64_t)u * a.max_parts * G * (D + 2);
  if (threadIdx.x < G) {
    const int j = threadIdx.x;
    float M = -INFINITY;
    for (int c = 0; c < n_parts; ++c) M = fmaxf(M, part[(c * G + j) * (D + 2) + D]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int c = 0; c < n_parts; ++c) {
        const float* pc = part + (c * G + j) * (D + 2);
        L = fmaf(pc[D + 1], ex2(pc[D] - M), L);
      }
    s_M[j] = M;
    s_invL[j] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  for (int x = threadIdx.x; x < G * D; x += blockDim.x) {
    const int j = x / D, d = x % D;
    const float M = s_M[j];
    float v = 0.f;
    if (M != -INFINITY)
      for (int c = 0; c < n_parts; ++c) {
        const float* pc = part + (c * G + j) * (D + 2);
        v = fmaf(pc[d], ex2(pc[D] - M), v);
      }
    v *= s_invL[j];
    T* op = out + ((int64_t)b * kv.Hq + g * G + j) * D + d;
    if constexpr (sizeof(T) == 2) *op = __float2bfloat16_rn(v);
    else *op = v;
  }
  if (acc != nullptr && a.logits != nullptr) {
    // eight entries per thread per round, every load of a round issued before
    // the first use (an entry's G logits as vector loads), so a round costs
    // one memory latency rather than eight
    const int ctx = kv.ctx_len[b];
    const int n_view = min(view_entries(a, ctx), a.max_entries);
    const float* lg = a.logits + ((int64_t)b * kv.Hkv + g) * a.max_entries * G;
    float* ar = acc + ((int64_t)b * kv.Hkv + g) * acc_stride;
    constexpr int U = 8;
    for (int e0 = threadIdx.x; e0 < n_view; e0 += U * blockDim.x) {
      int sl[U];
      float lv[U][G], old[U];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        const int e = e0 + k * blockDim.x;
        sl[k] = e < n_view ? view_slot(a, b, g, e, ctx) : -1;
        load_logits<G>(lg + (int64_t)e * G, sl[k] >= 0, lv[k]);
        old[k] = sl[k] >= 0 ? __ldcg(ar + sl[k]) : 0.f;
      }
#pragma unroll
      for (int k = 0; k < U; ++k) {
        float ps = 0.f;
#pragma unroll
        for (int j = 0; j < G; ++j) ps += ex2(lv[k][j] - s_M[j]) * s_invL[j];
        if (sl[k] >= 0) ar[sl[k]] = old[k] + ps;
      }
    }
  }
}

// End of a segment of unit u in CTA c: combines the 8 half-warp states
// (s_m, s_l, s_o, written before the call and fenced by a barrier) into the
// segment's partial, counts the segment and, in the last CTA to finish a
// segment of u, merges u.  Ends with a barrier.
template <typename T, int D, int G>
SE_DEV void finish_segment(const DecodeArgs& a, int u, int c, float (*s_m)[G], float (*s_l)[G],
                           float (*s_o)[G][D]) {
  __shared__ int s_last;
  int first, n_parts;
  unit_parts(a, u, &first, &n_parts);
  float* part = a.part + ((int64_t)u * a.max_parts + (c - first)) * G * (D + 2);
  for (int x = threadIdx.x; x < G * D; x += 128) {
    const int j = x / D, d = x % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 8; ++w) M = fmaxf(M, s_m[w][j]);
    float acc = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float f = ex2(s_m[w][j] - M);
        acc = fmaf(s_o[w][j][d], f, acc);
        L = fmaf(s_l[w][j], f, L);
      }
    }
    part[j * (D + 2) + d] = acc;
    if (d == 0) {
      part[j * (D + 2) + D] = M;
      part[j * (D + 2) + D + 1] = L;
    }
  }
  // the barrier orders the CTA's partial before thread 0's device-scope fence
  // and count; the last CTA's fence orders the count before its reads
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int last = atomicAdd(a.done + u, 1) == n_parts - 1;
    if (last) __threadfence();
    s_last = last;
  }
  __syncthreads();
  if (s_last) merge_chunks<T, D, G>(a, u, n_parts);
  // every segment of u has been counted: the counter is left at zero for
  // the next call on this workspace
  if (s_last && threadIdx.x == 0) a.done[u] = 0;
  __syncthreads();
}

// grid: n_cta; 128 threads = 8 half-warps.  Fallback for shapes whose stages
// do not fit shared memory: K and V rows are loaded straight into registers.
//
// A half-warp takes E = 16/G consecutive view entries per iteration; lane t
// owns dims [V t, V t + V) of K, V, q and o (V = D/16).  The E x G partial dot
// products of a lane are reduced across the 16 lanes by a 4-step xor
// reduce-scatter that leaves lane t with the complete logit of
// (entry t / G, head t % G): 15 shuffles per iteration instead of 4 G per
// entry.  Each lane then runs the base-2 online softmax for its own logit
// (one exponential), the per-head maxima are exchanged among the lanes of a
// head, the probabilities are all-gathered through shared memory, and every
// lane accumulates p * v for its dims.  o is rescaled only when a head's
// maximum grows.
template <typename T, int D, int G>
__global__ void __launch_bounds__(128) decode_partial_regs_kernel(DecodeArgs a) {
  pdl_enter();
  constexpr int V = D / 16;        // dims per lane
  constexpr int E = 16 / G;        // entries per half-warp iteration
  constexpr int SE = 8 * E;        // entries per slice
  static_assert(E * G == 16, "G must divide 16");
  __shared__ float s_p[8][16];
  __shared__ float s_m[8][G], s_l[8][G];
  __shared__ float s_o[8][G][D];
  const int c = blockIdx.x;
  const se_paged_kv& kv = a.kv;
  const int P = kv.page_size;
  const int hw = threadIdx.x >> 4, t = threadIdx.x & 15;
  const int my_e = t / G, my_h = t % G;   // the logit this lane holds after the reduction
  const float qscale = kLog2e * rsqrtf((float)D);
  const T* kp = static_cast<const T*>(kv.k_pool);
  const T* vp = static_cast<const T*>(kv.v_pool);
  const unsigned full = 0xffffffffu;
  const int64_t x0 = range_start(a, c), x1 = range_end(a, c);

  for (int64_t xs = x0; xs < x1;) {
    const int u = (int)(xs / a.sp);
    const int64_t xe = min(x1, (int64_t)(u + 1) * a.sp);
    const int b = u / kv.Hkv, g = u % kv.Hkv;
    const int ctx = kv.ctx_len[b];
    const int n_view = min(view_entries(a, ctx), a.max_entries);
    const int e_begin = (int)(xs - (int64_t)u * a.sp) * SE;
    const int e_end = min((int)(xe - (int64_t)u * a.sp) * SE, n_view);

    float q[G][V];
    const T* qb = static_cast<const T*>(a.q) + ((int64_t)b * kv.Hq + g * G) * D + t * V;
#pragma unroll
    for (int j = 0; j < G; ++j) {
      load_row<T, V>(qb + (int64_t)j * D, q[j]);
#pragma unroll
      for (int i = 0; i < V; ++i) q[j][i] *= qscale;
    }
    float m[G], o[G][V];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      m[j] = -INFINITY;
#pragma unroll
      for (int i = 0; i < V; ++i) o[j][i] = 0.f;
    }
    float l_own = 0.f;                 // running sum of this lane's head, own entries
    const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
    float* lg = a.logits ? a.logits + (int64_t)u * a.max_entries * G : nullptr;

    for (int base = e_begin; base < e_end; base += SE) {
      const int e0 = base + hw * E;
      float kf[E][V], vf[E][V];
      bool valid[E];
#pragma unroll
      for (int uu = 0; uu < E; ++uu) {
        const int e = e0 + uu;
        const int slot = e < e_end ? view_slot(a, b, g, e, ctx) : -1;
        const int page = slot >= 0 ? bt[slot / P] : -1;
        valid[uu] = page >= 0 && page < kv.num_pages;
        if (valid[uu]) {
          const int64_t off = (((int64_t)page * kv.Hkv + g) * P + slot % P) * D + t * V;
          load_row<T, V>(kp + off, kf[uu]);
          load_row<T, V>(vp + off, vf[uu]);
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) { kf[uu][i] = 0.f; vf[uu][i] = 0.f; }
        }
      }
      // partial dots, value index uu * G + j
      float part[16];
#pragma unroll
      for (int uu = 0; uu < E; ++uu)
#pragma unroll
        for (int j = 0; j < G; ++j) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < V; ++i) acc = fmaf(q[j][i], kf[uu][i], acc);
          part[uu * G + j] = acc;
        }
      // reduce-scatter: the lane keeps the upper half where its bit is set, so
      // after 4 steps lane t holds value t
#pragma unroll
      for (int step = 0; step < 4; ++step) {
        const int off = 8 >> step;
        const int n = 8 >> step;
        const bool upper = (t & off) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
          const float lo = part[i], hi = part[i + n];
          part[i] = (upper ? hi : lo) + __shfl_xor_sync(full, upper ? lo : hi, off);
        }
      }
      bool ok = false;
#pragma unroll
      for (int uu = 0; uu < E; ++uu) ok = (uu == my_e) ? valid[uu] : ok;
      const float sv = ok ? part[0] : -INFINITY;
      if (lg != nullptr && ok) lg[(int64_t)(e0 + my_e) * G + my_h] = sv;
      // maximum of this head over the iteration's entries: lanes of one head
      // differ in the bits above log2(G)
      float tmax = sv;
#pragma unroll
      for (int off = 8; off >= G; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(full, tmax, off));
      float m_mine = m[0];             // running max of my head before this iteration
#pragma unroll
      for (int j = 1; j < G; ++j) m_mine = (j == my_h) ? m[j] : m_mine;
      const float mn_mine = fmaxf(m_mine, tmax);
      const float alpha_mine =
          (mn_mine == -INFINITY || mn_mine == m_mine) ? 1.f : ex2(m_mine - mn_mine);
      const float p = (sv == -INFINITY) ? 0.f : ex2(sv - mn_mine);
      l_own = fmaf(l_own, alpha_mine, p);
      s_p[hw][t] = p;
      // every lane needs every head's new maximum / rescale factor
      bool grew = false;
      float alpha[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float mj = __shfl_sync(full, mn_mine, (threadIdx.x & 16) + j);
        alpha[j] = __shfl_sync(full, alpha_mine, (threadIdx.x & 16) + j);
        grew |= mj != m[j];
        m[j] = mj;
      }
      __syncwarp();
      if (grew) {
#pragma unroll
        for (int j = 0; j < G; ++j)
#pragma unroll
          for (int i = 0; i < V; ++i) o[j][i] *= alpha[j];
      }
#pragma unroll
      for (int uu = 0; uu < E; ++uu) {
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float pu = s_p[hw][uu * G + j];
#pragma unroll
          for (int i = 0; i < V; ++i) o[j][i] = fmaf(pu, vf[uu][i], o[j][i]);
        }
      }
      __syncwarp();
    }
    // running sums of each head: lanes of a head add up their own entries
    float lsum = l_own;
#pragma unroll
    for (int off = 8; off >= G; off >>= 1) lsum += __shfl_xor_sync(full, lsum, off);
    if (t < G) {
      float mt = m[0];
#pragma unroll
      for (int j = 1; j < G; ++j) mt = (j == t) ? m[j] : mt;
      s_m[hw][t] = mt;
      s_l[hw][t] = lsum;
    }
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
      for (int i = 0; i < V; ++i) s_o[hw][j][t * V + i] = o[j][i];
    __syncthreads();
    finish_segment<T, D, G>(a, u, c, s_m, s_l, s_o);
    xs = xe;
  }
}

// V elements of a K or V row in shared memory, as fp32.
template <typename T, int V>
SE_DEV void load_row_smem(const T* r, float* f) {
  if constexpr (sizeof(T) == 2 && V == 8) {
    unpack8_bf16(*reinterpret_cast<const uint4*>(r), f);
  } else {
#pragma unroll
    for (int i = 0; i < V; ++i) f[i] = (float)r[i];
  }
}

constexpr int kMaxChunk = 1024;   // view entries per CTA at most (see make_split)

template <typename T, int D, int G>
struct StagedGeom {
  static constexpr int V = D / 16;                 // dims per lane
  static constexpr int E = 16 / G;                 // entries per half-warp per stage
  static constexpr int SE = 8 * E;                 // entries per stage
  static constexpr int RB = D * (int)sizeof(T);    // bytes per K (or V) row
  static constexpr int STAGE_BYTES = SE * RB * 2;
  // three 16 KB stages keep four CTAs (sixteen warps) on an SM at 128 registers a thread
  static constexpr int STAGES =
      STAGE_BYTES <= 8192 ? 4 : (STAGE_BYTES <= 16384 ? 3 : (STAGE_BYTES <= 32768 ? 2 : 0));
  static constexpr int SMEM = STAGES * STAGE_BYTES + 128;   // + alignment of the stages to 128 B
  // CTAs an SM holds by shared memory (about 6 KB static besides SMEM),
  // at most four; eight heads a group take two (their q and o fill the
  // registers)
  static constexpr int MIN_CTAS =
      G >= 8 ? 2 : ((227 * 1024) / (SMEM + 6 * 1024) >= 4 ? 4 : 3);
};

// Issues the copies of one stage (segment entries [s0, s0 + SE)); called by
// all 32 lanes of one warp.  rows[x] is the K/V row of segment entry x in the
// pool ((page * Hkv + g) * P + row in page), -1 for none, resolved once per
// CTA.  A maximal run of entries that are consecutive rows of one page
// becomes one K and one V copy, issued by the lane that starts it.  valid[u]
// records whether entry u has a row (read by the consumers after the stage's
// barrier completes).  Lane 0 arrives on the barrier last.
template <typename T, int D, int G>
SE_DEV void issue_stage(const DecodeArgs& a, int s0, int n_seg, const int32_t* rows, uint8_t* dst,
                        uint64_t* bar, int8_t* valid, int lane) {
  using Gm = StagedGeom<T, D, G>;
  const int P = a.kv.page_size;
  const char* kp = static_cast<const char*>(a.kv.k_pool);
  const char* vp = static_cast<const char*>(a.kv.v_pool);
#pragma unroll
  for (int u0 = 0; u0 < Gm::SE; u0 += 32) {
    const int u = u0 + lane;
    const int x = s0 + u;
    const int prow = (u < Gm::SE && x < n_seg) ? rows[x] : -1;
    const bool ok = prow >= 0;
    if (u < Gm::SE) valid[u] = ok ? 1 : 0;
    // a run continues when this entry is the next row of the previous one's page
    const int prev = __shfl_up_sync(0xffffffffu, prow, 1);
    const bool cont = ok && lane > 0 && prev >= 0 && prev + 1 == prow && prow % P != 0;
    const uint32_t okm = __ballot_sync(0xffffffffu, ok);
    const uint32_t starts = __ballot_sync(0xffffffffu, ok && !cont);
    if (ok && !cont) {
      const uint32_t above = lane == 31 ? 0u : (~0u << (lane + 1));
      const uint32_t stop = (starts | ~okm) & above;
      const int end = stop ? __ffs(stop) - 1 : 32;
      const int len = end - lane;
      const int64_t off = (int64_t)prow * Gm::RB;
      tc::bulk_g2s(dst + u * Gm::RB, kp + off, (uint32_t)(len * Gm::RB), bar);
      tc::bulk_g2s(dst + Gm::SE * Gm::RB + u * Gm::RB, vp + off, (uint32_t)(len * Gm::RB), bar);
    }
  }
  __syncwarp();
  if (lane == 0) tc::mbar_arrive(bar);
}

// Copies the rows of one landed stage out to the pool: entry x of the stage
// (x < n) goes to K/V row dst[x] of the pool, none where dst[x] < 0.  Called
// by all 32 lanes of one warp: a maximal run of consecutive destination rows
// (within 32 entries) becomes one K and one V bulk store, issued by the lane
// that starts it; every lane then closes its bulk group (empty for most).
template <typename T, int D, int G>
SE_DEV void store_stage(const DecodeArgs& a, const uint8_t* stage, const int32_t* dst, int n,
                        int lane) {
  using Gm = StagedGeom<T, D, G>;
  char* kp = static_cast<char*>(a.kv.k_pool);
  char* vp = static_cast<char*>(a.kv.v_pool);
#pragma unroll
  for (int x0 = 0; x0 < Gm::SE; x0 += 32) {
    const int x = x0 + lane;
    const int d = x < n ? dst[x] : -1;
    const int prev = __shfl_up_sync(0xffffffffu, d, 1);
    const bool ok = d >= 0;
    const bool cont = ok && lane > 0 && prev >= 0 && prev + 1 == d;
    const uint32_t okm = __ballot_sync(0xffffffffu, ok);
    const uint32_t starts = __ballot_sync(0xffffffffu, ok && !cont);
    if (ok && !cont) {
      const uint32_t above = lane == 31 ? 0u : (~0u << (lane + 1));
      const uint32_t stop = (starts | ~okm) & above;
      const int len = (stop ? __ffs(stop) - 1 : 32) - lane;
      const uint32_t bytes = (uint32_t)(len * Gm::RB);
      tc::bulk_s2g(kp + (int64_t)d * Gm::RB, stage + x * Gm::RB, bytes);
      tc::bulk_s2g(vp + (int64_t)d * Gm::RB, stage + Gm::SE * Gm::RB + x * Gm::RB, bytes);
    }
  }
  tc::bulk_commit();
}

// Shared memory of the staged kernels: the stage ring and the per-half-warp
// softmax states.
template <int G, int SE>
struct StageRing {
  uint8_t* stages;       // STAGES buffers (K rows, then V rows), 128-byte aligned
  uint64_t* full;        // [STAGES] the copies of a stage have landed
  uint64_t* empty;       // [STAGES] the four warps are done with a stage
  int8_t (*valid)[SE];   // [4][SE] whether entry x of a stage has a row
  float (*p)[16];        // [8][16] probabilities of one iteration
  float (*m)[G];         // [8][G] half-warp maxima
  float (*l)[G];         // [8][G] half-warp sums
  int* abort;            // a wait ran out
};

// K/V row in the pool ((page * Hkv + g) * P + row in page) of view entries
// [e_begin, e_begin + n) of unit u, -1 for an entry past the view or without
// a resident row, written to rows[0, n) by the CTA's threads.  In the dense
// view the block-table reads do not wait for ctx_len (only the mask does).
// Returns how many of the n entries lie in the view.
SE_DEV int resolve_rows(const DecodeArgs& a, int u, int e_begin, int n, int32_t* rows) {
  const se_paged_kv& kv = a.kv;
  const int b = u / kv.Hkv, g = u % kv.Hkv;
  const int P = kv.page_size;
  const int ctx = kv.ctx_len[b];
  const int n_view = min(view_entries(a, ctx), a.max_entries);
  const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
  // four entries per thread per round, every load of a round issued before
  // the first use
  constexpr int R = 4;
  for (int x0 = threadIdx.x; x0 < n; x0 += R * blockDim.x) {
    int slot[R], page[R];
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const int x = x0 + k * blockDim.x;
      const int e = e_begin + x;
      if (a.view == SE_VIEW_DENSE) {
        const int ip = e / P;
        page[k] = (x < n && ip < kv.max_pages_per_seq) ? bt[ip] : -1;
        slot[k] = (x < n && e < n_view) ? e : -1;
      } else {
        slot[k] = (x < n && e < n_view) ? view_slot(a, b, g, e, ctx) : -1;
      }
    }
    if (a.view != SE_VIEW_DENSE) {
#pragma unroll
      for (int k = 0; k < R; ++k) page[k] = slot[k] >= 0 ? bt[slot[k] / P] : -1;
    }
#pragma unroll
    for (int k = 0; k < R; ++k) {
      const int x = x0 + k * blockDim.x;
      if (x < n)
        rows[x] = (slot[k] >= 0 && page[k] >= 0 && page[k] < kv.num_pages)
                      ? (page[k] * kv.Hkv + g) * P + slot[k] % P
                      : -1;
    }
  }
  return max(min(e_begin + n, n_view) - e_begin, 0);
}

// Streams view entries [e_begin, e_begin + n_seg) of unit u = (b, g), whose
// K/V rows are rows[0, n_seg), through the stage ring.  Warp 0 keeps
// STAGES-1 stages of copies in flight; every half-warp reads its E rows of
// each stage from shared memory (16 lanes x 16 bytes = one 256-byte row,
// conflict-free) and runs the reduce-scatter / online-softmax arithmetic of
// the register kernel above.  gi / gc count the stages the CTA has issued /
// consumed (stage n uses buffer n % STAGES), so buffers and barrier phases
// carry over from one call to the next.  On return the 8 half-warp states
// are in r.m, r.l and, as float [8][G][D], over the stage memory (every
// stage is idle by then), and all threads have passed a barrier.  A wait
// that runs out sets the status word and *r.abort and ends the stream; the
// states are then meaningless but the call still returns normally.
// COPY: every landed stage is also copied out to the pool rows dst[0, n_seg)
// (store_stage, by warp 0); a buffer is refilled, and the stage memory
// reused, only after those stores have read it (every lane of warp 0 waits
// for its own bulk groups).
template <typename T, int D, int G, bool COPY = false>
SE_DEV void stream_segment(const DecodeArgs& a, const StageRing<G, StagedGeom<T, D, G>::SE>& r,
                           int u, int e_begin, int n_seg, const int32_t* rows, int& gi, int& gc,
                           const int32_t* dst = nullptr) {
  using Gm = StagedGeom<T, D, G>;
  constexpr int V = Gm::V, E = Gm::E, SE = Gm::SE, RB = Gm::RB, S = Gm::STAGES;
  constexpr int V2 = V / 2;
  constexpr uint64_t kLimit = 2000000000ull;
  const se_paged_kv& kv = a.kv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hw = threadIdx.x >> 4, t = threadIdx.x & 15;
  const int my_e = t / G, my_h = t % G;
  const unsigned full_mask = 0xffffffffu;
  const bool producer = warp == 0;   // the whole warp issues, lane 0 arrives
  const float qscale = kLog2e * rsqrtf((float)D);
  const int b = u / kv.Hkv, g = u % kv.Hkv;
  const int n_it = cdiv(n_seg, SE);
  const int g0 = gi;   // stage count at the segment's start
  uint8_t* const stages = r.stages;

  // the first STAGES-1 stages; a buffer last used by an earlier segment is
  // refilled only after its consumers have released it
  if (producer) {
    for (int i = 0; i < min(S - 1, n_it); ++i) {
      const int n = g0 + i;
      const bool free_ok = n < S || tc::mbar_wait(&r.empty[n % S], ((n / S) - 1) & 1, kLimit);
      if (!__all_sync(full_mask, free_ok)) {
        if (lane == 0) {
          set_status(kv.status, SE_ERR_TIMEOUT);
          atomicExch(r.abort, 1);
        }
        break;
      }
      if constexpr (COPY) {
        tc::bulk_wait_read();
        __syncwarp();
      }
      issue_stage<T, D, G>(a, i * SE, n_seg, rows, stages + (n % S) * Gm::STAGE_BYTES,
                           &r.full[n % S], r.valid[n % S], lane);
      ++gi;
    }
  }

  float q[G][V];
  const T* qb = static_cast<const T*>(a.q) + ((int64_t)b * kv.Hq + g * G) * D + t * V;
#pragma unroll
  for (int j = 0; j < G; ++j) {
    load_row<T, V>(qb + (int64_t)j * D, q[j]);
#pragma unroll
    for (int i = 0; i < V; ++i) q[j][i] *= qscale;
  }
  // q and o as fp32 pairs: dot products and p * v updates run as paired FMAs
  uint64_t q2[G][V2], o2[G][V2];
  float m[G];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    m[j] = -INFINITY;
#pragma unroll
    for (int i = 0; i < V2; ++i) {
      q2[j][i] = tc::f2(q[j][2 * i], q[j][2 * i + 1]);
      o2[j][i] = 0;
    }
  }
  float l_own = 0.f;
  float* lg = a.logits ? a.logits + (int64_t)u * a.max_entries * G : nullptr;

  for (int it = 0; it < n_it; ++it) {
    if (producer && gi - g0 < n_it) {
      // refill the buffer consumed in the previous iteration
      const int n = gi;
      const bool free_ok = n < S || tc::mbar_wait(&r.empty[n % S], ((n / S) - 1) & 1, kLimit);
      if (__all_sync(full_mask, free_ok)) {
        if constexpr (COPY) {
          tc::bulk_wait_read();   // the stores of the buffer's last stage
          __syncwarp();
        }
        issue_stage<T, D, G>(a, (n - g0) * SE, n_seg, rows, stages + (n % S) * Gm::STAGE_BYTES,
                             &r.full[n % S], r.valid[n % S], lane);
        ++gi;
      } else if (lane == 0) {
        set_status(kv.status, SE_ERR_TIMEOUT);
        atomicExch(r.abort, 1);
      }
    }
    const int s = gc % S;
    const bool ok_wait = tc::mbar_wait(&r.full[s], (gc / S) & 1, kLimit);
    if (!__all_sync(full_mask, ok_wait)) {
      if (lane == 0) {
        set_status(kv.status, SE_ERR_TIMEOUT);
        atomicExch(r.abort, 1);
      }
      break;
    }
    const uint8_t* kst = stages + s * Gm::STAGE_BYTES;
    const uint8_t* vst = kst + SE * RB;
    if constexpr (COPY) {
      if (warp == 0) store_stage<T, D, G>(a, kst, dst + it * SE, min(SE, n_seg - it * SE), lane);
    }
    const int e0 = e_begin + it * SE + hw * E;
    // K rows are read from the stage one entry at a time; V rows are read
    // again after the probabilities are known (the stage is released after)
    bool valid[E];
    float part[16];
#pragma unroll
    for (int uu = 0; uu < E; ++uu) {
      valid[uu] = r.valid[s][hw * E + uu] != 0;
      float kf[V];
      if (valid[uu]) {
        load_row_smem<T, V>(reinterpret_cast<const T*>(kst + (hw * E + uu) * RB) + t * V, kf);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) kf[i] = 0.f;
      }
      uint64_t k2[V2];
#pragma unroll
      for (int i = 0; i < V2; ++i) k2[i] = tc::f2(kf[2 * i], kf[2 * i + 1]);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        uint64_t acc2 = 0;
#pragma unroll
        for (int i = 0; i < V2; ++i) acc2 = tc::ffma2(q2[j][i], k2[i], acc2);
        float lo, hi;
        tc::f2split(acc2, lo, hi);
        part[uu * G + j] = lo + hi;
      }
    }
#pragma unroll
    for (int step = 0; step < 4; ++step) {
      const int off = 8 >> step;
      const int n = 8 >> step;
      const bool upper = (t & off) != 0;
#pragma unroll
      for (int i = 0; i < n; ++i) {
        const float lo = part[i], hi = part[i + n];
        part[i] = (upper ? hi : lo) + __shfl_xor_sync(full_mask, upper ? lo : hi, off);
      }
    }
    bool ok = false;
#pragma unroll
    for (int uu = 0; uu < E; ++uu) ok = (uu == my_e) ? valid[uu] : ok;
    const float sv = ok ? part[0] : -INFINITY;
    if (lg != nullptr && ok) lg[(int64_t)(e0 + my_e) * G + my_h] = sv;
    float tmax = sv;
#pragma unroll
    for (int off = 8; off >= G; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(full_mask, tmax, off));
    float m_mine = m[0];
#pragma unroll
    for (int j = 1; j < G; ++j) m_mine = (j == my_h) ? m[j] : m_mine;
    const float mn_mine = fmaxf(m_mine, tmax);
    const float alpha_mine =
        (mn_mine == -INFINITY || mn_mine == m_mine) ? 1.f : ex2(m_mine - mn_mine);
    const float p = (sv == -INFINITY) ? 0.f : ex2(sv - mn_mine);
    l_own = fmaf(l_own, alpha_mine, p);
    r.p[hw][t] = p;
    bool grew = false;
    float alpha[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float mj = __shfl_sync(full_mask, mn_mine, (threadIdx.x & 16) + j);
      alpha[j] = __shfl_sync(full_mask, alpha_mine, (threadIdx.x & 16) + j);
      grew |= mj != m[j];
      m[j] = mj;
    }
    __syncwarp();
    if (grew) {
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const uint64_t a2 = tc::f2(alpha[j], alpha[j]);
#pragma unroll
        for (int i = 0; i < V2; ++i) o2[j][i] = tc::ffma2(o2[j][i], a2, 0);
      }
    }
#pragma unroll
    for (int uu = 0; uu < E; ++uu) {
      float vf[V];
      if (valid[uu]) {
        load_row_smem<T, V>(reinterpret_cast<const T*>(vst + (hw * E + uu) * RB) + t * V, vf);
      } else {
#pragma unroll
        for (int i = 0; i < V; ++i) vf[i] = 0.f;
      }
      uint64_t v2[V2];
#pragma unroll
      for (int i = 0; i < V2; ++i) v2[i] = tc::f2(vf[2 * i], vf[2 * i + 1]);
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float pu = r.p[hw][uu * G + j];
        const uint64_t p2 = tc::f2(pu, pu);
#pragma unroll
        for (int i = 0; i < V2; ++i) o2[j][i] = tc::ffma2(p2, v2[i], o2[j][i]);
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&r.empty[s]);   // done with this stage's rows
    ++gc;
  }
  // drain: after a timeout, copies of the last stages may still be in flight
  // (each earlier stage was waited on before its buffer was refilled)
  if (producer && lane == 0)
    for (int i = max(0, gi - S); i < gi; ++i) tc::mbar_wait(&r.full[i % S], (i / S) & 1, kLimit);
  if constexpr (COPY) {
    if (producer) tc::bulk_wait_read();   // the stage memory is reused below
  }
  float lsum = l_own;
#pragma unroll
  for (int off = 8; off >= G; off >>= 1) lsum += __shfl_xor_sync(full_mask, lsum, off);
  if (t < G) {
    float mt = m[0];
#pragma unroll
    for (int j = 1; j < G; ++j) mt = (j == t) ? m[j] : mt;
    r.m[hw][t] = mt;
    r.l[hw][t] = lsum;
  }
  __syncthreads();   // every stage of the segment has been read: reuse the stage memory
  float (*s_o)[G][D] = reinterpret_cast<float (*)[G][D]>(stages);
#pragma unroll
  for (int j = 0; j < G; ++j)
#pragma unroll
    for (int i = 0; i < V2; ++i) {
      float lo, hi;
      tc::f2split(o2[j][i], lo, hi);
      s_o[hw][j][t * V + 2 * i] = lo;
      s_o[hw][j][t * V + 2 * i + 1] = hi;
    }
  __syncthreads();
}

// grid: n_cta; 128 threads = 8 half-warps; dynamic smem StagedGeom::SMEM.
// Warp 0 keeps STAGES-1 stages of copies in flight within a segment; every
// half-warp reads its E rows of each stage from shared memory (16 lanes x 16
// bytes = one 256-byte row, conflict-free) and runs the same reduce-scatter /
// online-softmax arithmetic as the register kernel above.  Stage buffers and
// barrier phases follow a count of the stages the CTA has issued, so they
// carry over from one segment to the next; at a segment's end the stages are
// idle and hold the half-warp states while they are combined.
// The stream of a segment is the one stream_segment runs for the cluster
// kernels, written out here: built from stream_segment, this kernel measured
// about 5 % slower on the multi-wave grids it serves (same instructions,
// scheduled differently by the compiler).
template <typename T, int D, int G>
__global__ void __launch_bounds__(128, StagedGeom<T, D, G>::MIN_CTAS) decode_partial_kernel(DecodeArgs a) {
  pdl_enter();
  using Gm = StagedGeom<T, D, G>;
  constexpr int V = Gm::V, E = Gm::E, SE = Gm::SE, RB = Gm::RB, S = Gm::STAGES;
  extern __shared__ __align__(1024) uint8_t dsmem[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 127) & ~uintptr_t(127));
  __shared__ uint64_t full[4], empty[4];
  __shared__ int8_t s_valid[4][SE];
  __shared__ int32_t s_rows[kMaxChunk];   // K/V row of each entry of the CTA's range, -1 for none
  __shared__ float s_p[8][16];
  __shared__ float s_m[8][G], s_l[8][G];
  __shared__ int s_nseg[kMaxChunk / SE];   // viewed entries of each segment of the range
  __shared__ int s_abort;
  static_assert(S * Gm::STAGE_BYTES >= 8 * G * D * 4, "merge buffer must fit the stages");
  const int c = blockIdx.x;
  const se_paged_kv& kv = a.kv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hw = threadIdx.x >> 4, t = threadIdx.x & 15;
  const int my_e = t / G, my_h = t % G;
  const unsigned full_mask = 0xffffffffu;
  constexpr uint64_t kLimit = 2000000000ull;
  const int64_t x0 = range_start(a, c), x1 = range_end(a, c);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 4);
    }
    tc::fence_barrier_init();
  }
  // resolve every entry of the range to its K/V row once (view -> slot ->
  // block table), segment by segment, so the stage producer only reads
  // shared memory; s_nseg keeps each segment's count of viewed entries
  for (int64_t xs = x0, k = 0; xs < x1; ++k) {
    const int u = (int)(xs / a.sp);
    const int64_t xe = min(x1, (int64_t)(u + 1) * a.sp);
    const int e_begin = (int)(xs - (int64_t)u * a.sp) * SE;
    const int n = resolve_rows(a, u, e_begin, (int)(xe - xs) * SE, s_rows + (int)(xs - x0) * SE);
    if (threadIdx.x == 0) s_nseg[k] = n;
    xs = xe;
  }
  __syncthreads();
  const bool producer = warp == 0;   // the whole warp issues, lane 0 arrives
  const float qscale = kLog2e * rsqrtf((float)D);
  constexpr int V2 = V / 2;
  int gi = 0;   // stages issued by this CTA (stage n uses buffer n % S)
  int gc = 0;   // stages consumed

  for (int64_t xs = x0, k = 0; xs < x1; ++k) {
    const int u = (int)(xs / a.sp);
    const int64_t xe = min(x1, (int64_t)(u + 1) * a.sp);
    const int b = u / kv.Hkv, g = u % kv.Hkv;
    const int e_begin = (int)(xs - (int64_t)u * a.sp) * SE;
    const int n_seg = s_nseg[k];
    const int n_it = cdiv(n_seg, SE);
    const int32_t* rows = s_rows + (int)(xs - x0) * SE;
    const int g0 = gi;   // stage count at the segment's start

    // the first STAGES-1 stages; a buffer last used by an earlier segment is
    // refilled only after its consumers have released it
    if (producer) {
      for (int i = 0; i < min(S - 1, n_it); ++i) {
        const int n = g0 + i;
        const bool free_ok = n < S || tc::mbar_wait(&empty[n % S], ((n / S) - 1) & 1, kLimit);
        if (!__all_sync(full_mask, free_ok)) {
          if (lane == 0) {
            set_status(kv.status, SE_ERR_TIMEOUT);
            atomicExch(&s_abort, 1);
          }
          break;
        }
        issue_stage<T, D, G>(a, i * SE, n_seg, rows, stages + (n % S) * Gm::STAGE_BYTES,
                             &full[n % S], s_valid[n % S], lane);
        ++gi;
      }
    }

    float q[G][V];
    const T* qb = static_cast<const T*>(a.q) + ((int64_t)b * kv.Hq + g * G) * D + t * V;
#pragma unroll
    for (int j = 0; j < G; ++j) {
      load_row<T, V>(qb + (int64_t)j * D, q[j]);
#pragma unroll
      for (int i = 0; i < V; ++i) q[j][i] *= qscale;
    }
    // q and o as fp32 pairs: dot products and p * v updates run as paired FMAs
    uint64_t q2[G][V2], o2[G][V2];
    float m[G];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      m[j] = -INFINITY;
#pragma unroll
      for (int i = 0; i < V2; ++i) {
        q2[j][i] = tc::f2(q[j][2 * i], q[j][2 * i + 1]);
        o2[j][i] = 0;
      }
    }
    float l_own = 0.f;
    float* lg = a.logits ? a.logits + (int64_t)u * a.max_entries * G : nullptr;

    for (int it = 0; it < n_it; ++it) {
      if (producer && gi - g0 < n_it) {
        // refill the buffer consumed in the previous iteration
        const int n = gi;
        const bool free_ok = n < S || tc::mbar_wait(&empty[n % S], ((n / S) - 1) & 1, kLimit);
        if (__all_sync(full_mask, free_ok)) {
          issue_stage<T, D, G>(a, (n - g0) * SE, n_seg, rows, stages + (n % S) * Gm::STAGE_BYTES,
                               &full[n % S], s_valid[n % S], lane);
          ++gi;
        } else if (lane == 0) {
          set_status(kv.status, SE_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
        }
      }
      const int s = gc % S;
      const bool ok_wait = tc::mbar_wait(&full[s], (gc / S) & 1, kLimit);
      if (!__all_sync(full_mask, ok_wait)) {
        if (lane == 0) {
          set_status(kv.status, SE_ERR_TIMEOUT);
          atomicExch(&s_abort, 1);
        }
        break;
      }
      const uint8_t* kst = stages + s * Gm::STAGE_BYTES;
      const uint8_t* vst = kst + SE * RB;
      const int e0 = e_begin + it * SE + hw * E;
      // K rows are read from the stage one entry at a time; V rows are read
      // again after the probabilities are known (the stage is released after)
      bool valid[E];
      float part[16];
#pragma unroll
      for (int uu = 0; uu < E; ++uu) {
        valid[uu] = s_valid[s][hw * E + uu] != 0;
        float kf[V];
        if (valid[uu]) {
          load_row_smem<T, V>(reinterpret_cast<const T*>(kst + (hw * E + uu) * RB) + t * V, kf);
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) kf[i] = 0.f;
        }
        uint64_t k2[V2];
#pragma unroll
        for (int i = 0; i < V2; ++i) k2[i] = tc::f2(kf[2 * i], kf[2 * i + 1]);
#pragma unroll
        for (int j = 0; j < G; ++j) {
          uint64_t acc2 = 0;
#pragma unroll
          for (int i = 0; i < V2; ++i) acc2 = tc::ffma2(q2[j][i], k2[i], acc2);
          float lo, hi;
          tc::f2split(acc2, lo, hi);
          part[uu * G + j] = lo + hi;
        }
      }
#pragma unroll
      for (int step = 0; step < 4; ++step) {
        const int off = 8 >> step;
        const int n = 8 >> step;
        const bool upper = (t & off) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
          const float lo = part[i], hi = part[i + n];
          part[i] = (upper ? hi : lo) + __shfl_xor_sync(full_mask, upper ? lo : hi, off);
        }
      }
      bool ok = false;
#pragma unroll
      for (int uu = 0; uu < E; ++uu) ok = (uu == my_e) ? valid[uu] : ok;
      const float sv = ok ? part[0] : -INFINITY;
      if (lg != nullptr && ok) lg[(int64_t)(e0 + my_e) * G + my_h] = sv;
      float tmax = sv;
#pragma unroll
      for (int off = 8; off >= G; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(full_mask, tmax, off));
      float m_mine = m[0];
#pragma unroll
      for (int j = 1; j < G; ++j) m_mine = (j == my_h) ? m[j] : m_mine;
      const float mn_mine = fmaxf(m_mine, tmax);
      const float alpha_mine =
          (mn_mine == -INFINITY || mn_mine == m_mine) ? 1.f : ex2(m_mine - mn_mine);
      const float p = (sv == -INFINITY) ? 0.f : ex2(sv - mn_mine);
      l_own = fmaf(l_own, alpha_mine, p);
      s_p[hw][t] = p;
      bool grew = false;
      float alpha[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const float mj = __shfl_sync(full_mask, mn_mine, (threadIdx.x & 16) + j);
        alpha[j] = __shfl_sync(full_mask, alpha_mine, (threadIdx.x & 16) + j);
        grew |= mj != m[j];
        m[j] = mj;
      }
      __syncwarp();
      if (grew) {
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const uint64_t a2 = tc::f2(alpha[j], alpha[j]);
#pragma unroll
          for (int i = 0; i < V2; ++i) o2[j][i] = tc::ffma2(o2[j][i], a2, 0);
        }
      }
#pragma unroll
      for (int uu = 0; uu < E; ++uu) {
        float vf[V];
        if (valid[uu]) {
          load_row_smem<T, V>(reinterpret_cast<const T*>(vst + (hw * E + uu) * RB) + t * V, vf);
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) vf[i] = 0.f;
        }
        uint64_t v2[V2];
#pragma unroll
        for (int i = 0; i < V2; ++i) v2[i] = tc::f2(vf[2 * i], vf[2 * i + 1]);
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float pu = s_p[hw][uu * G + j];
          const uint64_t p2 = tc::f2(pu, pu);
#pragma unroll
          for (int i = 0; i < V2; ++i) o2[j][i] = tc::ffma2(p2, v2[i], o2[j][i]);
        }
      }
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&empty[s]);   // done with this stage's rows
      ++gc;
    }
    // drain: after a timeout, copies of the last stages may still be in flight
    // (each earlier stage was waited on before its buffer was refilled)
    if (producer && lane == 0)
      for (int i = max(0, gi - S); i < gi; ++i) tc::mbar_wait(&full[i % S], (i / S) & 1, kLimit);
    float lsum = l_own;
#pragma unroll
    for (int off = 8; off >= G; off >>= 1) lsum += __shfl_xor_sync(full_mask, lsum, off);
    if (t < G) {
      float mt = m[0];
#pragma unroll
      for (int j = 1; j < G; ++j) mt = (j == t) ? m[j] : mt;
      s_m[hw][t] = mt;
      s_l[hw][t] = lsum;
    }
    __syncthreads();   // every stage of the segment has been read: reuse the stage memory
    float (*s_o)[G][D] = reinterpret_cast<float (*)[G][D]>(stages);
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
      for (int i = 0; i < V2; ++i) {
        float lo, hi;
        tc::f2split(o2[j][i], lo, hi);
        s_o[hw][j][t * V + 2 * i] = lo;
        s_o[hw][j][t * V + 2 * i + 1] = hi;
      }
    __syncthreads();
    finish_segment<T, D, G>(a, u, c, s_m, s_l, s_o);
    // the stage memory was written and read as plain shared memory; order
    // that before the next segment's copies into it
    tc::fence_proxy_async_smem();
    __syncthreads();
    if (s_abort) break;
    xs = xe;
  }
}

constexpr int kMaxCluster = 16;   // CTAs of a unit in the cluster split (non-portable above 8)

// The merge of a cluster split (decode_cluster_kernel): combines the CTA's
// half-warp states (s_m, s_l, and o over the stage memory as left by
// stream_segment) into its partial, in place over the first half-warp's o;
// waits for the cluster; merges this CTA's G D / k elements of o from the
// peers' partials and writes them; arrives on the cluster barrier that ends
// the reads of the peers' shared memory (the caller waits on it before it
// leaves).  Leaves the unit's maximum and 1 / sum of each head in s_M, s_invL.
template <typename T, int D, int G>
SE_DEV void cluster_merge(const DecodeArgs& a, cg::cluster_group& cluster, int k, int rank, int b,
                          int g, uint8_t* stages, float (*s_m)[G], float (*s_l)[G], float* s_M,
                          float* s_invL) {
  constexpr int GD = G * D;
  static_assert(GD % kMaxCluster == 0, "o splits evenly over the cluster");
  __shared__ float s_pm[G], s_pl[G];                            // this CTA's partial: maxima, sums
  __shared__ float s_cm[kMaxCluster][G], s_ce[kMaxCluster][G];  // the peers' maxima; their weights
  const se_paged_kv& kv = a.kv;
  // the CTA's partial (each element is read and written by one thread)
  float (*s_o)[G][D] = reinterpret_cast<float (*)[G][D]>(stages);
  for (int x = threadIdx.x; x < GD; x += 128) {
    const int j = x / D, d = x % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 8; ++w) M = fmaxf(M, s_m[w][j]);
    float acc = 0.f, L = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float f = ex2(s_m[w][j] - M);
        acc = fmaf(s_o[w][j][d], f, acc);
        L = fmaf(s_l[w][j], f, L);
      }
    }
    s_o[0][j][d] = acc;
    if (d == 0) {
      s_pm[j] = M;
      s_pl[j] = L;
    }
  }
  cluster.sync();   // every partial of the unit is in its CTA's shared memory

  // this CTA's elements of o: tpe threads (adjacent lanes) per element, each
  // summing cpt = k / tpe of the partials (every tpe-th one), then a fixed
  // xor tree over the tpe lanes.  One round of peer reads fetches the
  // maxima and sums and every o value the thread needs.
  constexpr int NV = GD >= 128 ? GD / 128 : 1;   // o values per thread at most
  const int per = GD / k;
  int tpe = 1;
  while (tpe < k && tpe * 2 * per <= 128) tpe <<= 1;
  const int cpt = k / tpe, epr = 128 / tpe, rounds = cdiv(per, epr);
  const int sub = threadIdx.x & (tpe - 1);
  const float* po = &s_o[0][0][0];
  float ov[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int x = (i / cpt) * epr + threadIdx.x / tpe;
    ov[i] = (i < rounds * cpt && x < per)
                ? *cluster.map_shared_rank(po + rank * per + x, sub + (i % cpt) * tpe)
                : 0.f;
  }
  if (threadIdx.x < k * G) {
    const int c = threadIdx.x / G, j = threadIdx.x % G;
    s_cm[c][j] = *cluster.map_shared_rank(&s_pm[j], c);
    s_ce[c][j] = *cluster.map_shared_rank(&s_pl[j], c);
  }
  __syncthreads();
  if (threadIdx.x < G) {
    const int j = threadIdx.x;
    float M = -INFINITY;
    for (int c = 0; c < k; ++c) M = fmaxf(M, s_cm[c][j]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int c = 0; c < k; ++c) L = fmaf(s_ce[c][j], ex2(s_cm[c][j] - M), L);
    s_M[j] = M;
    s_invL[j] = L > 0.f ? 1.f / L : 0.f;
  }
  __syncthreads();
  if (threadIdx.x < k * G) {
    const int c = threadIdx.x / G, j = threadIdx.x % G;
    s_ce[c][j] = s_M[j] == -INFINITY ? 0.f : ex2(s_cm[c][j] - s_M[j]);
  }
  __syncthreads();
  T* out = static_cast<T*>(a.out);
  for (int rd = 0; rd < rounds; ++rd) {
    const int x = rd * epr + threadIdx.x / tpe;
    const bool ok = x < per;
    const int xg = rank * per + (ok ? x : 0);
    const int j = xg / D, d = xg % D;
    float v = 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (i / cpt == rd) v = fmaf(ov[i], s_ce[sub + (i % cpt) * tpe][j], v);
    for (int off = 1; off < tpe; off <<= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (ok && sub == 0) {
      v *= s_invL[j];
      T* op = out + ((int64_t)b * kv.Hq + g * G + j) * D + d;
      if constexpr (sizeof(T) == 2) *op = __float2bfloat16_rn(v);
      else *op = v;
    }
  }
  // the peers' shared memory is no longer read by this CTA
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

// grid: units x k CTAs in clusters of k = a.k_cl (a power of two up to 16);
// 128 threads; dynamic smem StagedGeom::SMEM.  Cluster u is unit u = (b, g);
// its CTA of rank r streams slices [r sp / k, (r + 1) sp / k) of the unit and
// combines its half-warp states into one partial (m, l, o) in its own shared
// memory.  After a cluster barrier every CTA reads the k maxima and sums from
// its peers' shared memory, merges its own G D / k elements of o from the
// peers' partials (the partials of an element are summed in a fixed order,
// so the result does not depend on timing), writes them, and for H2O adds
// sum_h p_{h,j} to the running score of each of its own entries from the
// logits it stored.  A second cluster barrier keeps every CTA's shared
// memory alive until its peers have read it.  Every thread of every CTA
// reaches both barriers, also after a stage wait has run out.
template <typename T, int D, int G>
__global__ void __launch_bounds__(128, StagedGeom<T, D, G>::MIN_CTAS) decode_cluster_kernel(DecodeArgs a) {
  using Gm = StagedGeom<T, D, G>;
  constexpr int SE = Gm::SE, S = Gm::STAGES;
  static_assert(S * Gm::STAGE_BYTES >= 8 * G * D * 4, "merge buffer must fit the stages");
  extern __shared__ __align__(1024) uint8_t dsmem[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 127) & ~uintptr_t(127));
  __shared__ uint64_t full[4], empty[4];
  __shared__ int8_t s_valid[4][SE];
  __shared__ int32_t s_rows[kMaxChunk];
  __shared__ float s_p[8][16];
  __shared__ float s_m[8][G], s_l[8][G];
  __shared__ int s_abort;
  const StageRing<G, SE> ring{stages, full, empty, s_valid, s_p, s_m, s_l, &s_abort};
  cg::cluster_group cluster = cg::this_cluster();
  const se_paged_kv& kv = a.kv;
  const int k = a.k_cl;
  const int rank = (int)cluster.block_rank();
  const int u = blockIdx.x / k;
  const int b = u / kv.Hkv, g = u % kv.Hkv;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 4);
    }
    tc::fence_barrier_init();
  }
  pdl_enter();
  const int xs = (int)((int64_t)rank * a.sp / k), xe = (int)((int64_t)(rank + 1) * a.sp / k);
  const int e_begin = xs * SE;
  const int n_seg = resolve_rows(a, u, e_begin, (xe - xs) * SE, s_rows);
  __syncthreads();
  int gi = 0, gc = 0;
  stream_segment<T, D, G>(a, ring, u, e_begin, n_seg, s_rows, gi, gc);

  __shared__ float s_M[G], s_invL[G];
  cluster_merge<T, D, G>(a, cluster, k, rank, b, g, stages, s_m, s_l, s_M, s_invL);

  if (a.acc != nullptr && a.logits != nullptr) {
    // the running scores of this CTA's own entries, from the logits it
    // stored; four entries per thread per round, the loads of a round issued
    // before the first use
    const int ctx = kv.ctx_len[b];
    const int e_end = e_begin + n_seg;
    const float* lg = a.logits + (int64_t)u * a.max_entries * G;
    float* ar = a.acc + (int64_t)u * a.acc_stride;
    constexpr int U = 4;
    for (int e00 = e_begin + threadIdx.x; e00 < e_end; e00 += U * 128) {
      int sl[U];
      float lv[U][G], old[U];
#pragma unroll
      for (int kk = 0; kk < U; ++kk) {
        const int e = e00 + kk * 128;
        sl[kk] = (e < e_end && s_rows[e - e_begin] >= 0) ? view_slot(a, b, g, e, ctx) : -1;
        load_logits<G>(lg + (int64_t)e * G, sl[kk] >= 0, lv[kk]);
        old[kk] = sl[kk] >= 0 ? __ldcg(ar + sl[kk]) : 0.f;
      }
#pragma unroll
      for (int kk = 0; kk < U; ++kk) {
        float ps = 0.f;
#pragma unroll
        for (int j = 0; j < G; ++j) ps += ex2(lv[kk][j] - s_M[j]) * s_invL[j];
        if (sl[kk] >= 0) ar[sl[kk]] = old[kk] + ps;
      }
    }
  }
  __syncwarp();
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Compaction into fresh pages fused with decode attention over the result
// ---------------------------------------------------------------------------

constexpr int kMaxChunkCD = 512;   // entries per CTA of the fused kernel

struct CompactDecodeArgs {
  DecodeArgs d;                // the cache before the call; the dense view of the result
  const int32_t* keep;         // [B][Hkv][keep_stride] kept slots, ascending
  int32_t keep_stride;
  const int32_t* first_slot;   // [B]
  const float* aux;            // [B][Hkv][aux_stride] values that move with the entries, or null
  int64_t aux_stride;
  CompactWs w;                 // the plan (compact_plan_kernel) and the staging for the commit
};

// Entries [e_begin, e_begin + n) of unit u in the compacted sequence: the K/V
// row each is read from (its old page), the row it is written to (its fresh
// page; -1 below the first rewritten block, where the entry stays), and the
// staged slot-map / aux values of the rewritten ones -- the same sources,
// destinations and checks as the gather kernel of a plain compaction.  A
// sequence longer than the view (max_entries) is refused like a bad keep
// index: status SE_ERR_BOUNDS, and the commit does not run.  Returns how many
// of the n entries lie in the compacted sequence.
SE_DEV int resolve_compact_rows(const CompactDecodeArgs& ca, int u, int e_begin, int n,
                                int32_t* rows, int32_t* dst) {
  const se_paged_kv& kv = ca.d.kv;
  const CompactWs& w = ca.w;
  const int b = u / kv.Hkv, h = u % kv.Hkv;
  const int P = kv.page_size;
  const int pb = w.pb[b], fs = ca.first_slot[b], nctx = w.new_ctx[b], octx = w.old_ctx[b];
  const int pop0 = w.ctrl->top0 - 1 - w.off_new[b];
  if (nctx > ca.d.max_entries) {
    if (threadIdx.x == 0) {
      set_status(kv.status, SE_ERR_BOUNDS);
      atomicExch(&w.ctrl->abort, 1);
    }
    return 0;
  }
  const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
  const int32_t* keep = ca.keep + (int64_t)u * ca.keep_stride;
  const int64_t smax = (int64_t)kv.max_pages_per_seq * P;
  const int64_t tb = (int64_t)u * w.row;
  bool bad = false;
  for (int x = threadIdx.x; x < n; x += blockDim.x) {
    const int e = e_begin + x;
    int src = -1, drow = -1;
    if (e < nctx) {
      if (e < pb * P) {
        src = e;
      } else {
        src = e < fs ? e : keep[e - fs];
        if (e >= fs && !(src >= fs && src < octx && (e == fs || src > keep[e - fs - 1]))) {
          bad = true;
          src = -1;
        } else {
          const int dp = kv.free_list[pop0 - (e / P - pb)];
          if (dp < 0 || dp >= kv.num_pages) {
            bad = true;
            src = -1;
          } else {
            drow = (dp * kv.Hkv + h) * P + e % P;
            w.slot_tmp[tb + (e - pb * P)] = kv.slot_map[(int64_t)u * smax + src];
            if (ca.aux != nullptr && w.aux_tmp != nullptr)
              w.aux_tmp[tb + (e - pb * P)] = ca.aux[(int64_t)u * ca.aux_stride + src];
          }
        }
      }
    }
    const int page = src >= 0 ? bt[src / P] : -1;
    if (src >= 0 && (page < 0 || page >= kv.num_pages)) bad = true;
    const bool ok = src >= 0 && page >= 0 && page < kv.num_pages;
    rows[x] = ok ? (page * kv.Hkv + h) * P + src % P : -1;
    dst[x] = ok ? drow : -1;
  }
  if (bad) {
    set_status(kv.status, SE_ERR_BOUNDS);
    atomicExch(&w.ctrl->abort, 1);
  }
  return max(min(e_begin + n, nctx) - e_begin, 0);
}

// grid: units x k CTAs in clusters of k = d.k_cl; 128 threads; dynamic smem
// StagedGeom::SMEM.  The cluster decode kernel over the dense view of the
// compacted cache, reading every entry from where it lies before the call:
// each landed stage of rewritten entries is also stored to the entries' rows
// in their fresh pages, so the kept K/V cross HBM once on the way in and once
// on the way out.  The CTAs of (b, head 0) record sequence b's fresh pages
// for the commit.  After a planning error nothing is read or written (the
// output is then undefined and the status word says why).
template <typename T, int D, int G>
__global__ void __launch_bounds__(128, StagedGeom<T, D, G>::MIN_CTAS)
compact_decode_kernel(CompactDecodeArgs ca) {
  using Gm = StagedGeom<T, D, G>;
  constexpr int SE = Gm::SE, S = Gm::STAGES;
  static_assert(S * Gm::STAGE_BYTES >= 8 * G * D * 4, "merge buffer must fit the stages");
  const DecodeArgs& a = ca.d;
  extern __shared__ __align__(1024) uint8_t dsmem[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(dsmem) + 127) & ~uintptr_t(127));
  __shared__ uint64_t full[4], empty[4];
  __shared__ int8_t s_valid[4][SE];
  __shared__ int32_t s_rows[kMaxChunkCD], s_dst[kMaxChunkCD];
  __shared__ float s_p[8][16];
  __shared__ float s_m[8][G], s_l[8][G];
  __shared__ int s_abort;
  __shared__ float s_M[G], s_invL[G];
  const StageRing<G, SE> ring{stages, full, empty, s_valid, s_p, s_m, s_l, &s_abort};
  cg::cluster_group cluster = cg::this_cluster();
  const se_paged_kv& kv = a.kv;
  const int k = a.k_cl;
  const int rank = (int)cluster.block_rank();
  const int u = blockIdx.x / k;
  const int b = u / kv.Hkv, g = u % kv.Hkv;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < S; ++i) {
      tc::mbar_init(&full[i], 1);
      tc::mbar_init(&empty[i], 4);
    }
    tc::fence_barrier_init();
  }
  pdl_enter();
  const bool planned = ca.w.ctrl->abort == 0;
  const int xs = (int)((int64_t)rank * a.sp / k), xe = (int)((int64_t)(rank + 1) * a.sp / k);
  const int e_begin = xs * SE;
  const int n_seg = planned ? resolve_compact_rows(ca, u, e_begin, (xe - xs) * SE, s_rows, s_dst) : 0;
  __syncthreads();
  int gi = 0, gc = 0;
  stream_segment<T, D, G, true>(a, ring, u, e_begin, n_seg, s_rows, gi, gc, s_dst);
  // the cluster of (b, head 0) records sequence b's fresh pages, one share
  // per CTA (after the stream, off its critical start)
  if (planned && g == 0) record_fresh_pages(kv, ca.w, b, rank, k);
  cluster_merge<T, D, G>(a, cluster, k, rank, b, g, stages, s_m, s_l, s_M, s_invL);
  if (threadIdx.x < 32) tc::bulk_wait_all();   // the copies have reached global memory
  __syncwarp();
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

struct DecodeWs {
  float* part;
  float* logits;
  int32_t* done;
};

struct DecodeSplit {
  int sp;          // slices per unit
  int64_t ts;      // slices in all
  int n_cta;
  int k_al, w_al;  // aligned split (k_al = 0: stream split)
  int max_parts;   // partial slots per unit
  int k_cl;        // cluster split: CTAs per unit, 0 where it does not apply
};

// CTA slots of the staged kernel on GB300: 152 SMs x 4 resident CTAs.
constexpr int kCtaSlots = 152 * 4;

// Aligned chunks: about four CTAs per SM, at least 128 entries (64 KB of
// bf16 K/V at d = 128) per CTA so that set-up and the partial write stay
// small next to the stream, at most kMaxChunk, evened out over the unit.
// They are used when all of them run at once or when they make four waves or
// more (a ragged last wave costs little then); otherwise the stream split
// cuts the slices into whole waves of ranges, again of at most kMaxChunk and
// at least 128 entries.  Depends on the shape only (the workspace size does).
static DecodeSplit make_split(const se_paged_kv* kv, int max_entries) {
  const int G = max(kv->Hq / max(kv->Hkv, 1), 1);
  const int SE = max(128 / G, 1);
  const int64_t units = std::max<int64_t>((int64_t)kv->B * kv->Hkv, 1);
  const int me = max(max_entries, 1);
  DecodeSplit d;
  d.sp = cdiv(me, SE);
  d.ts = units * d.sp;
  int chunk = kMaxChunk;
  while (chunk > 128 && units * cdiv(me, chunk) < kCtaSlots) chunk >>= 1;
  chunk = min(chunk, cdiv(cdiv(me, cdiv(me, chunk)), 128) * 128);
  const int w = max(chunk / SE, 1);
  const int k = cdiv(d.sp, w);
  const int64_t n_al = units * k;
  // cluster split: the most CTAs per unit (a power of two up to 16) that
  // keep every CTA within kMaxChunk entries and the grid within one wave of
  // four CTAs per SM.  Grids of several waves keep the split-K forms: there
  // the merge is a small share of the time, and clusters of 16 leave SMs of
  // a GPC unused.
  d.k_cl = 0;
  const int64_t w_cl = max(kMaxChunk / SE, 1);
  for (int kc = 1; kc <= kMaxCluster; kc *= 2) {
    if (cdiv64(d.sp, kc) > w_cl) continue;
    if (units * kc > kCtaSlots) break;
    d.k_cl = kc;
  }
  if (n_al <= kCtaSlots || n_al >= 4 * kCtaSlots) {
    d.n_cta = (int)n_al;
    d.k_al = k;
    d.w_al = w;
    d.max_parts = k;
    return d;
  }
  const int w_max = max(kMaxChunk / SE, 1), w_min = max(128 / SE, 1);
  int64_t n = cdiv64(cdiv64(d.ts, w_max), kCtaSlots) * kCtaSlots;
  if (d.ts / n < w_min) n = std::max<int64_t>(1, d.ts / w_min);
  d.n_cta = (int)n;
  d.k_al = 0;
  d.w_al = 0;
  d.max_parts = (int)cdiv64(d.sp, d.ts / n) + 1;
  return d;
}

static DecodeWs carve_decode(const se_paged_kv* kv, int max_entries, const DecodeSplit& sp,
                             void* ws, size_t* bytes) {
  WsCarver c(ws);
  DecodeWs w;
  const int G = max(kv->Hq / max(kv->Hkv, 1), 1);
  const size_t units = (size_t)kv->B * kv->Hkv;
  w.part = c.take<float>(units * sp.max_parts * G * (kv->D + 2));
  w.logits = c.take<float>(units * max_entries * G);
  w.done = c.take<int32_t>(units);
  *bytes = c.bytes();
  return w;
}

// Whether clusters of k CTAs of `kernel` (128 threads, `smem` bytes of
// dynamic shared memory) fit the current device; asked once per device and
// cluster size.  known[dev] holds bit log2(k) once asked and bit 8 + log2(k)
// when they fit.
static bool cluster_fits(const void* kernel, int smem, int k, std::atomic<uint32_t>* known) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  int bit = 0;
  while ((1 << bit) < k) ++bit;
  const uint32_t v = known[dev].load(std::memory_order_acquire);
  if (v & (1u << bit)) return (v >> (8 + bit)) & 1u;
  bool ok = k <= 8 ||
            cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (ok) {
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)k;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(k);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    ok = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n > 0;
  }
  if (!ok) (void)cudaGetLastError();   // a refused query is an answer, not a launch error
  known[dev].fetch_or((1u << bit) | (ok ? 1u << (8 + bit) : 0u), std::memory_order_acq_rel);
  return ok;
}

template <typename T, int D, int G>
static void launch_decode_t(const DecodeArgs& a, cudaStream_t st) {
  using Gm = StagedGeom<T, D, G>;
  const dim3 grid(a.n_cta);
  bool staged = Gm::STAGES > 0;
  if constexpr (Gm::STAGES > 0) {
    if (a.k_cl > 0) {
      static std::atomic<uint64_t> attr_cl{0};
      static std::atomic<uint32_t> known[64];
      const void* kc = reinterpret_cast<const void*>(&decode_cluster_kernel<T, D, G>);
      if (allow_smem(kc, Gm::SMEM, attr_cl) && cluster_fits(kc, Gm::SMEM, a.k_cl, known)) {
        se_launch_cluster(decode_cluster_kernel<T, D, G>,
                          dim3((unsigned)(a.kv.B * a.kv.Hkv * a.k_cl)), 128, Gm::SMEM, st, a.k_cl, a);
        return;
      }
    }
    DecodeArgs ak = a;
    ak.k_cl = 0;
    static std::atomic<uint64_t> attr{0};
    staged = allow_smem(reinterpret_cast<const void*>(&decode_partial_kernel<T, D, G>), Gm::SMEM,
                        attr);
    if (staged) se_launch(decode_partial_kernel<T, D, G>, grid, 128, Gm::SMEM, st, ak);
  }
  if (!staged) se_launch(decode_partial_regs_kernel<T, D, G>, grid, 128, 0, st, a);
}

template <typename T, int D>
static se_status launch_decode_d(const DecodeArgs& a, int G, cudaStream_t st) {
  switch (G) {
    case 1: launch_decode_t<T, D, 1>(a, st); return SE_OK;
    case 2: launch_decode_t<T, D, 2>(a, st); return SE_OK;
    case 4: launch_decode_t<T, D, 4>(a, st); return SE_OK;
    case 8: launch_decode_t<T, D, 8>(a, st); return SE_OK;
    default: return SE_ERR_UNSUPPORTED;
  }
}

template <typename T, int D, int G>
static se_status launch_compact_decode_t(const CompactDecodeArgs& ca, cudaStream_t st) {
  using Gm = StagedGeom<T, D, G>;
  if constexpr (Gm::STAGES > 0) {
    static std::atomic<uint64_t> attr{0};
    static std::atomic<uint32_t> known[64];
    const void* kf = reinterpret_cast<const void*>(&compact_decode_kernel<T, D, G>);
    if (!allow_smem(kf, Gm::SMEM, attr) || !cluster_fits(kf, Gm::SMEM, ca.d.k_cl, known))
      return SE_ERR_UNSUPPORTED;
    se_launch_cluster(compact_decode_kernel<T, D, G>, dim3((unsigned)ca.d.n_cta), 128, Gm::SMEM, st,
                      ca.d.k_cl, ca);
    return SE_OK;
  }
  return SE_ERR_UNSUPPORTED;
}

template <typename T, int D>
static se_status launch_compact_decode_d(const CompactDecodeArgs& ca, int G, cudaStream_t st) {
  switch (G) {
    case 1: return launch_compact_decode_t<T, D, 1>(ca, st);
    case 2: return launch_compact_decode_t<T, D, 2>(ca, st);
    case 4: return launch_compact_decode_t<T, D, 4>(ca, st);
    case 8: return launch_compact_decode_t<T, D, 8>(ca, st);
    default: return SE_ERR_UNSUPPORTED;
  }
}

// Launches compact_decode_kernel between the plan and the commit of a
// compaction into fresh pages when the shape takes it: a staged kernel for
// the dtype, D and group size, a cluster of at most 16 CTAs of at most
// kMaxChunkCD entries per (sequence, KV head), and clusters that fit the
// device.  Returns SE_ERR_UNSUPPORTED, with nothing launched, otherwise.
se_status launch_compact_decode(const se_paged_kv* kv, const int32_t* keep, int32_t keep_stride,
                                const int32_t* first_slot, const float* aux, int64_t aux_stride,
                                const CompactWs& w, const void* q, void* o, int32_t max_entries,
                                cudaStream_t st) {
  const int G = kv->Hq / kv->Hkv;
  if (G < 1 || 128 % G != 0 || max_entries < 1) return SE_ERR_UNSUPPORTED;
  if ((int64_t)kv->num_pages * kv->Hkv * kv->page_size > INT32_MAX) return SE_ERR_UNSUPPORTED;
  const int SE = 128 / G;
  const int64_t units = (int64_t)kv->B * kv->Hkv;
  const int sp = cdiv(max_entries, SE);
  // the split of decode attention's cluster form (make_split), with at most
  // kMaxChunkCD entries per CTA
  int k = 0;
  for (int kc = 1; kc <= kMaxCluster; kc *= 2) {
    if (cdiv(sp, kc) * SE > kMaxChunkCD) continue;
    if (units * kc > kCtaSlots) break;
    k = kc;
  }
  if (k == 0) return SE_ERR_UNSUPPORTED;
  CompactDecodeArgs ca{};
  ca.d.kv = *kv;
  ca.d.q = q;
  ca.d.view = SE_VIEW_DENSE;
  ca.d.sp = sp;
  ca.d.ts = units * sp;
  ca.d.n_cta = (int)(units * k);
  ca.d.max_entries = max_entries;
  ca.d.out = o;
  ca.d.k_cl = k;
  ca.keep = keep;
  ca.keep_stride = keep_stride;
  ca.first_slot = first_slot;
  ca.aux = aux;
  ca.aux_stride = aux_stride;
  ca.w = w;
  if (kv->dtype == SE_BF16 && kv->D == 128) return launch_compact_decode_d<__nv_bfloat16, 128>(ca, G, st);
  if (kv->dtype == SE_BF16 && kv->D == 64) return launch_compact_decode_d<__nv_bfloat16, 64>(ca, G, st);
  if (kv->dtype == SE_F32 && kv->D == 128) return launch_compact_decode_d<float, 128>(ca, G, st);
  if (kv->dtype == SE_F32 && kv->D == 64) return launch_compact_decode_d<float, 64>(ca, G, st);
  return SE_ERR_UNSUPPORTED;
}

}  // namespace se

using namespace se;

extern "C" size_t se_sparse_decode_attn_workspace_size(const se_paged_kv* kv, int32_t max_entries) {
  if (kv == nullptr || max_entries < 0) return 0;
  size_t b = 0;
  carve_decode(kv, max_entries, make_split(kv, max_entries), nullptr, &b);
  return b;
}

// clear_counters: zero the per-unit segment counters before the launch (the
// library's own scratch array, which no caller can re-zero after an error);
// a caller's workspace is zero before its first use and every call that
// completes leaves the counters zero.
static se_status decode_attn(const se_paged_kv* kv, const void* q, int32_t view,
                             const int32_t* sel, int32_t sel_stride, int32_t n_sel,
                             int32_t max_entries, void* o, float* acc_scores, int64_t acc_stride,
                             void* workspace, size_t workspace_bytes, void* stream,
                             bool clear_counters) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (q == nullptr || o == nullptr || workspace == nullptr || max_entries < 1) return SE_ERR_INVALID_ARG;
  if (view != SE_VIEW_DENSE && (sel == nullptr || n_sel < 0 || sel_stride < n_sel))
    return SE_ERR_INVALID_ARG;
  if (view < SE_VIEW_DENSE || view > SE_VIEW_TOKENS) return SE_ERR_INVALID_ARG;
  const int G = kv->Hq / kv->Hkv;
  // K/V rows of the pool are indexed with 32-bit integers in the kernels
  if ((int64_t)kv->num_pages * kv->Hkv * kv->page_size > INT32_MAX) return SE_ERR_UNSUPPORTED;
  const DecodeSplit sp = make_split(kv, max_entries);
  if ((sp.k_al > 0 ? sp.w_al : cdiv64(sp.ts, sp.n_cta)) * (128 / G) > kMaxChunk)
    return SE_ERR_UNSUPPORTED;
  size_t need = 0;
  DecodeWs w = carve_decode(kv, max_entries, sp, workspace, &need);
  if (workspace_bytes < need) return SE_ERR_INVALID_ARG;
  DecodeArgs a{*kv, q, view, sel, sel_stride, n_sel, sp.sp, sp.ts, sp.n_cta, sp.k_al, sp.w_al,
               sp.max_parts,
               w.part, acc_scores ? w.logits : nullptr, max_entries, o, acc_scores, acc_stride,
               w.done, sp.k_cl};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (clear_counters &&
      cudaMemsetAsync(w.done, 0, sizeof(int32_t) * kv->B * kv->Hkv, st) != cudaSuccess)
    return SE_ERR_CUDA;
  if (kv->dtype == SE_BF16 && kv->D == 128) s = launch_decode_d<__nv_bfloat16, 128>(a, G, st);
  else if (kv->dtype == SE_BF16 && kv->D == 64) s = launch_decode_d<__nv_bfloat16, 64>(a, G, st);
  else if (kv->dtype == SE_F32 && kv->D == 128) s = launch_decode_d<float, 128>(a, G, st);
  else if (kv->dtype == SE_F32 && kv->D == 64) s = launch_decode_d<float, 64>(a, G, st);
  else return SE_ERR_UNSUPPORTED;
  if (s != SE_OK) return s;
  return se_last_launch_status();
}

extern "C" se_status se_sparse_decode_attn(const se_paged_kv* kv, const void* q, int32_t view,
                                           const int32_t* sel, int32_t sel_stride, int32_t n_sel,
                                           int32_t max_entries, void* o, float* acc_scores,
                                           int64_t acc_stride, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  return decode_attn(kv, q, view, sel, sel_stride, n_sel, max_entries, o, acc_scores, acc_stride,
                     workspace, workspace_bytes, stream, false);
}

// ---------------------------------------------------------------------------
// Allocation-free variant: scratch in a fixed device array owned by the
// library (see se_sparse_decode_attn_static in se.h for who needs it).
// ---------------------------------------------------------------------------

#include <mutex>

static __device__ __align__(256) unsigned char g_decode_static_scratch[SE_DECODE_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (cudaGetSymbolAddress, with that device current).  The host-side
// name of the array is only a stand-in and must never reach a kernel.
se_status static_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_static_scratch) != cudaSuccess || p == nullptr)
      return SE_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SE_OK;
}

}  // namespace

extern "C" se_status se_sparse_decode_attn_static(const se_paged_kv* kv, const void* q,
                                                  int32_t view, const int32_t* sel,
                                                  int32_t sel_stride, int32_t n_sel,
                                                  int32_t max_entries, void* o, float* acc_scores,
                                                  int64_t acc_stride, void* stream) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (max_entries < 1) return SE_ERR_INVALID_ARG;
  if (se_sparse_decode_attn_workspace_size(kv, max_entries) > SE_DECODE_STATIC_SCRATCH_BYTES)
    return SE_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  s = static_scratch(&scratch);
  if (s != SE_OK) return s;
  return decode_attn(kv, q, view, sel, sel_stride, n_sel, max_entries, o, acc_scores, acc_stride,
                     scratch, SE_DECODE_STATIC_SCRATCH_BYTES, stream, true);
}
