// Quest decode step in one launch: page bounds, top pages + the current page,
// and attention over the selected pages.
//
// SparseEngine "What it is" / "How it works" (Quest: a query-aware page
// selection from per-page key min / max, then attention over the selected
// pages through the AttentionView).  Same results as se_quest_page_select
// followed by se_sparse_decode_attn over the page view; this form removes the
// round trips through global memory and the launches between the steps.
//
// One thread-block cluster of 8 CTAs per (sequence b, KV head g):
//   1. bounds   CTA r owns an eighth of the full pages 0 .. nb-2.  Half-warps
//               read kmin / kmax rows (16 bytes a lane, eight pages in flight)
//               and compute U = sum_{h in g} sum_i max(q_i kmax_i, q_i kmin_i)
//               into order-preserving integer keys in shared memory.
//   2. select   every CTA radix-selects its local top pages (ties: lower page
//               first); the global top set lies inside the union of the local
//               ones, so CTA 0 gathers the 8 local lists (already in ascending
//               page order) through distributed shared memory and selects
//               again.  The current page nb-1 is appended.
//   3. attend   every CTA reads the final list from CTA 0 and runs the online
//               softmax over its share of the selected pages (half-warp per
//               16/G entries, xor reduce-scatter of the G dot products, as in
//               the decode kernel); CTA 0 merges the 8 partials and writes o.
// Cluster barriers separate the phases; no CTA leaves while a peer may still
// read its shared memory.
#include <cooperative_groups.h>

#include "se_common.cuh"

namespace se {

namespace {

constexpr int kQfCtas = 8;                       // CTAs per cluster
constexpr int kQfThreads = 256;
constexpr int kQfItems = 8;                      // candidate pages per thread
constexpr int kQfCap = kQfThreads * kQfItems;    // candidate pages per CTA
constexpr int kQfMaxTop = 256;                   // selected pages per (b, g), current included
constexpr int kQfGather = 8;                     // keys per thread in CTA 0's final select
constexpr int kQfAttnWarps = 8;                  // warps of phase 3

struct QfArgs {
  se_paged_kv kv;
  const __nv_bfloat16* kmin;
  const __nv_bfloat16* kmax;
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  int32_t* page_idx;      // [B][Hkv][top + 1] or null
  int32_t* n_sel;         // [B] or null
  int top;
};

// k-th largest of the keys held by the CTA (ITEMS per thread, key 0 = absent):
// up to three radix rounds of 11, 11 and 10 bits, fewer when every key under
// the prefix found so far is taken.  Returns the threshold T on the digits
// resolved (mask TM) and how many keys whose resolved digits equal T are
// taken (the lowest-indexed ones).
template <int ITEMS>
SE_DEV void block_kth_key(const uint32_t (&key)[ITEMS], int kk, int* hist, int* tmp, int* s_digit,
                          int* s_rem, uint32_t& T, uint32_t& TM, int& need_eq) {
  const int tid = threadIdx.x;
  uint32_t prefix = 0, pmask = 0;
  int remaining = kk;
  if (kk > 0) {
#pragma unroll 1
    for (int round = 0; round < 3; ++round) {
      const int shift = round == 0 ? 21 : (round == 1 ? 10 : 0);
      const int nbins = round == 2 ? 1024 : 2048;
      const uint32_t dmask = (uint32_t)nbins - 1u;
      for (int i = tid; i < nbins; i += blockDim.x) hist[i] = 0;
      __syncthreads();
      hist_add_keys<ITEMS>(hist, key, shift, dmask, pmask, prefix);
      __syncthreads();
      radix_find_digit(hist, nbins, remaining, tmp, s_digit, s_rem);
      prefix |= (uint32_t)*s_digit << shift;
      remaining = *s_rem;
      pmask |= dmask << shift;
      const bool whole_bin = hist[*s_digit] == remaining;
      __syncthreads();
      if (whole_bin) break;
    }
  }
  T = kk > 0 ? prefix : 0xffffffffu;
  TM = kk > 0 ? pmask : 0xffffffffu;
  need_eq = kk > 0 ? remaining : 0;
}

// Selection flags for the k largest keys (ties: lower index, i.e. lower
// thread / item first) and each selected key's rank in index order.
template <int ITEMS>
SE_DEV int block_select(const uint32_t (&key)[ITEMS], int kk, int* hist, int* tmp, int* s_digit,
                        int* s_rem, bool (&sel)[ITEMS], int* total) {
  uint32_t T, TM;
  int need_eq;
  block_kth_key<ITEMS>(key, kk, hist, tmp, s_digit, s_rem, T, TM, need_eq);
  int c_eq = 0;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) c_eq += (key[i] != 0u && (key[i] & TM) == T) ? 1 : 0;
  int dummy;
  int eq_rank = block_exclusive_scan(c_eq, tmp, &dummy);
  int c_sel = 0;
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
    c_sel += sel[i] ? 1 : 0;
  }
  return block_exclusive_scan(c_sel, tmp, total);
}

template <int G>
struct QfSmem {
  uint32_t key[kQfCap];                      // bound keys of this CTA's pages
  int32_t phys[kQfCap];                      // their physical pages (phase 1);
                                             // the selected ones' (phase 3)
  int hist[2048];
  int tmp[33];
  int digit;
  int rem;
  int loc_n;
  uint32_t loc_key[kQfMaxTop];               // local top, ascending page order
  int32_t loc_page[kQfMaxTop];
  uint32_t all_key[kQfCtas * kQfMaxTop];     // CTA 0: the gathered local tops
  int32_t all_page[kQfCtas * kQfMaxTop];
  int peer_n[kQfCtas];                       // CTA 0: local list sizes
  int sel_n;                                 // CTA 0: final list (read by peers)
  int32_t sel_page[kQfMaxTop];
  int my_n;                                  // this CTA's share of the list
  int32_t my_page[kQfMaxTop];
  float p[2 * kQfAttnWarps][16];             // phase 3 probabilities per half-warp
  float hm[2 * kQfAttnWarps][G], hl[2 * kQfAttnWarps][G];
  float ho[2 * kQfAttnWarps][G][128];
  float cm[G], cl[G];                        // this CTA's merged partial
  float all_m[kQfCtas * G], all_l[kQfCtas * G];  // CTA 0: every CTA's (m, l)
  float co[G][128];
};

template <int G>
__global__ void __cluster_dims__(kQfCtas, 1, 1) __launch_bounds__(kQfThreads, 1)
quest_fused_kernel(QfArgs a) {
  pdl_enter();
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int D = 128, V = 8, E = 16 / G;
  extern __shared__ __align__(16) uint8_t qf_raw[];
  QfSmem<G>& sm = *reinterpret_cast<QfSmem<G>*>(qf_raw);
  const se_paged_kv& kv = a.kv;
  const int rank = (int)cluster.block_rank();
  const int g = blockIdx.x / kQfCtas, b = blockIdx.y, tid = threadIdx.x;
  const int P = kv.page_size;
  const int ctx = kv.ctx_len[b];
  const int nb = cdiv(max(ctx, 0), P);
  const int n_cand = max(nb - 1, 0);                  // full pages compete
  const int per = cdiv(n_cand, kQfCtas);
  // the same for every CTA of the cluster: all return before the first barrier
  if (ctx < 0 || per > kQfCap || nb > kv.max_pages_per_seq) {
    if (rank == 0 && tid == 0) set_status(kv.status, SE_ERR_BOUNDS);
    return;
  }
  const int c0 = min(rank * per, n_cand), c1 = min(c0 + per, n_cand), n_loc = c1 - c0;
  const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
  const int lane = tid & 31, hw = tid >> 4, t = tid & 15;

  // ---- phase 1: page bounds ----
  for (int i = tid; i < n_loc; i += kQfThreads) sm.phys[i] = bt[c0 + i];
  for (int i = tid; i < kQfCap; i += kQfThreads) sm.key[i] = 0u;
  __syncthreads();
  // max(q kmax, q kmin) = max(q, 0) kmax + min(q, 0) kmin: two FMAs per term
  float qp[G][V], qn[G][V];
#pragma unroll
  for (int j = 0; j < G; ++j) {
    const uint4 u = ldg_nc_v4(a.q + ((int64_t)b * kv.Hq + g * G + j) * D + t * V);
    float qv[V];
    unpack8_bf16(u, qv);
#pragma unroll
    for (int i = 0; i < V; ++i) {
      qp[j][i] = fmaxf(qv[i], 0.f);
      qn[j][i] = fminf(qv[i], 0.f);
    }
  }
  bool bad_page = false;
  // rounds of kInFlight pages per half-warp; the next round's rows load while
  // the current round is reduced
  constexpr int kInFlight = 8, kRound = kInFlight * (kQfThreads / 16);
  uint4 cmn[kInFlight], cmx[kInFlight];
  bool cok[kInFlight];
  auto load_round = [&](int base, uint4 (&mn)[kInFlight], uint4 (&mx)[kInFlight],
                        bool (&ok)[kInFlight]) {
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      const int i = base + u * (kQfThreads / 16) + hw;
      const int page = i < n_loc ? sm.phys[i] : -1;
      ok[u] = page >= 0 && page < kv.num_pages;
      bad_page |= i < n_loc && !ok[u];
      if (ok[u]) {
        const int64_t off = ((int64_t)page * kv.Hkv + g) * D + t * V;
        mn[u] = ldg_nc_v4(a.kmin + off);
        mx[u] = ldg_nc_v4(a.kmax + off);
      }
    }
  };
  if (n_loc > 0) load_round(0, cmn, cmx, cok);
  for (int base = 0; base < n_loc; base += kRound) {
    uint4 nmn[kInFlight], nmx[kInFlight];
    bool nok[kInFlight];
    if (base + kRound < n_loc) {
      load_round(base + kRound, nmn, nmx, nok);
    } else {
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) nok[u] = false;
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      float acc = 0.f;
      if (cok[u]) {
        float mn[V], mx[V];
        unpack8_bf16(cmn[u], mn);
        unpack8_bf16(cmx[u], mx);
#pragma unroll
        for (int j = 0; j < G; ++j) {
          float part = 0.f;
#pragma unroll
          for (int i = 0; i < V; ++i) part = fmaf(qn[j][i], mn[i], fmaf(qp[j][i], mx[i], part));
          acc += part;
        }
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      const int i = base + u * (kQfThreads / 16) + hw;
      if (cok[u] && t == 0) sm.key[i] = float_key(acc);
    }
#pragma unroll
    for (int u = 0; u < kInFlight; ++u) {
      cmn[u] = nmn[u];
      cmx[u] = nmx[u];
      cok[u] = nok[u];
    }
  }
  if (bad_page) set_status(kv.status, SE_ERR_BOUNDS);
  __syncthreads();

  // ---- phase 2a: local top pages ----
  const int top = min(a.top, kQfMaxTop - 1);
  {
    uint32_t key[kQfItems];
#pragma unroll
    for (int i = 0; i < kQfItems; ++i) key[i] = sm.key[tid * kQfItems + i];
    int n_valid = 0;
#pragma unroll
    for (int i = 0; i < kQfItems; ++i) n_valid += key[i] != 0u;
    int valid_total;
    block_exclusive_scan(n_valid, sm.tmp, &valid_total);
    bool sel[kQfItems];
    int total;
    int pos = block_select<kQfItems>(key, min(top, valid_total), sm.hist, sm.tmp, &sm.digit,
                                     &sm.rem, sel, &total);
#pragma unroll
    for (int i = 0; i < kQfItems; ++i)
      if (sel[i]) {
        sm.loc_key[pos] = key[i];
        sm.loc_page[pos] = c0 + tid * kQfItems + i;
        pos++;
      }
    if (tid == 0) sm.loc_n = total;
  }
  cluster.sync();                                     // local lists complete

  // ---- phase 2b: CTA 0 selects among the local tops ----
  if (rank == 0) {
    // warp r copies CTA r's local list (eight warps, eight CTAs)
    static_assert(kQfThreads / 32 == kQfCtas, "one warp per CTA of the cluster");
    if (tid < kQfCtas) sm.peer_n[tid] = cluster.map_shared_rank(&sm, tid)->loc_n;
    __syncthreads();
    const int w = tid >> 5;
    int off = 0, n_all = 0;
    for (int r = 0; r < kQfCtas; ++r) {
      off += r < w ? sm.peer_n[r] : 0;
      n_all += sm.peer_n[r];
    }
    {
      const QfSmem<G>* peer = cluster.map_shared_rank(&sm, w);
      for (int i = lane; i < sm.peer_n[w]; i += 32) {
        sm.all_key[off + i] = peer->loc_key[i];
        sm.all_page[off + i] = peer->loc_page[i];
      }
    }
    __syncthreads();
    uint32_t key[kQfGather];
#pragma unroll
    for (int i = 0; i < kQfGather; ++i) {
      const int x = tid * kQfGather + i;
      key[i] = x < n_all ? sm.all_key[x] : 0u;
    }
    bool sel[kQfGather];
    int total;
    int pos = block_select<kQfGather>(key, min(top, n_all), sm.hist, sm.tmp, &sm.digit,
                                      &sm.rem, sel, &total);
#pragma unroll
    for (int i = 0; i < kQfGather; ++i)
      if (sel[i]) sm.sel_page[pos++] = sm.all_page[tid * kQfGather + i];
    if (tid == 0) {
      int n = total;
      if (nb >= 1) sm.sel_page[n++] = nb - 1;          // the current page
      sm.sel_n = n;
    }
    __syncthreads();
    if (a.page_idx != nullptr) {
      int32_t* out = a.page_idx + ((int64_t)b * kv.Hkv + g) * (a.top + 1);
      for (int i = tid; i < a.top + 1; i += kQfThreads) out[i] = i < sm.sel_n ? sm.sel_page[i] : -1;
    }
    if (a.n_sel != nullptr && g == 0 && tid == 0) a.n_sel[b] = sm.sel_n;
  }
  cluster.sync();                                     // final list complete

  // ---- phase 3: attention over this CTA's share of the selected pages ----
  {
    const QfSmem<G>* lead = cluster.map_shared_rank(&sm, 0);
    const int n_sel = lead->sel_n;
    const int pp = cdiv(n_sel, kQfCtas);
    const int p0 = min(rank * pp, n_sel), p1 = min(p0 + pp, n_sel);
    for (int i = tid; i < p1 - p0; i += kQfThreads) {
      const int blk = lead->sel_page[p0 + i];
      sm.my_page[i] = blk;
      sm.phys[i] = (blk >= 0 && blk < nb) ? bt[blk] : -1;
    }
    if (tid == 0) sm.my_n = p1 - p0;
  }
  __syncthreads();
  const int n_ent = sm.my_n * P;
  {
    const float qscale = kLog2e * rsqrtf((float)D);
    float qs[G][V];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const uint4 u = ldg_nc_v4(a.q + ((int64_t)b * kv.Hq + g * G + j) * D + t * V);
      unpack8_bf16(u, qs[j]);
#pragma unroll
      for (int i = 0; i < V; ++i) qs[j][i] *= qscale;
    }
    const int my_e = t / G, my_h = t % G;
    float m[G], o[G][V];
#pragma unroll
    for (int j = 0; j < G; ++j) {
      m[j] = -INFINITY;
#pragma unroll
      for (int i = 0; i < V; ++i) o[j][i] = 0.f;
    }
    float l_own = 0.f;
    const __nv_bfloat16* kp = static_cast<const __nv_bfloat16*>(kv.k_pool);
    const __nv_bfloat16* vp = static_cast<const __nv_bfloat16*>(kv.v_pool);
    const unsigned full = 0xffffffffu;
    for (int base = 0; base < n_ent; base += 2 * kQfAttnWarps * E) {
      const int e0 = base + hw * E;
      float kf[E][V], vf[E][V];
      bool valid[E];
#pragma unroll
      for (int u = 0; u < E; ++u) {
        const int e = e0 + u;
        const int pi = e / P, row = e % P;
        const int page = e < n_ent ? sm.phys[pi] : -1;
        const int slot = e < n_ent ? sm.my_page[pi] * P + row : ctx;
        valid[u] = page >= 0 && page < kv.num_pages && slot < ctx;
        if (valid[u]) {
          const int64_t off = (((int64_t)page * kv.Hkv + g) * P + row) * D + t * V;
          unpack8_bf16(ldg_nc_v4(kp + off), kf[u]);
          unpack8_bf16(ldg_nc_v4(vp + off), vf[u]);
        } else {
#pragma unroll
          for (int i = 0; i < V; ++i) { kf[u][i] = 0.f; vf[u][i] = 0.f; }
        }
      }
      float part[16];
#pragma unroll
      for (int u = 0; u < E; ++u)
#pragma unroll
        for (int j = 0; j < G; ++j) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < V; ++i) acc = fmaf(qs[j][i], kf[u][i], acc);
          part[u * G + j] = acc;
        }
      // reduce-scatter: lane t ends with value t = (entry t / G, head t % G)
#pragma unroll
      for (int step = 0; step < 4; ++step) {
        const int off = 8 >> step;
        const bool upper = (t & off) != 0;
#pragma unroll
        for (int i = 0; i < (8 >> step); ++i) {
          const float lo = part[i], hi = part[i + (8 >> step)];
          part[i] = (upper ? hi : lo) + __shfl_xor_sync(full, upper ? lo : hi, off);
        }
      }
      bool okv = false;
#pragma unroll
      for (int u = 0; u < E; ++u) okv = (u == my_e) ? valid[u] : okv;
      const float sv = okv ? part[0] : -INFINITY;
      float tmax = sv;
#pragma unroll
      for (int off = 8; off >= G; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(full, tmax, off));
      float m_mine = m[0];
#pragma unroll
      for (int j = 1; j < G; ++j) m_mine = (j == my_h) ? m[j] : m_mine;
      const float mn_mine = fmaxf(m_mine, tmax);
      const float alpha_mine =
          (mn_mine == -INFINITY || mn_mine == m_mine) ? 1.f : exp2f(m_mine - mn_mine);
      const float pr = (sv == -INFINITY) ? 0.f : exp2f(sv - mn_mine);
      l_own = fmaf(l_own, alpha_mine, pr);
      sm.p[hw][t] = pr;
      float alpha[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        m[j] = __shfl_sync(full, mn_mine, (lane & 16) + j);
        alpha[j] = __shfl_sync(full, alpha_mine, (lane & 16) + j);
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < G; ++j)
#pragma unroll
        for (int i = 0; i < V; ++i) o[j][i] *= alpha[j];
#pragma unroll
      for (int u = 0; u < E; ++u)
#pragma unroll
        for (int j = 0; j < G; ++j) {
          const float pu = sm.p[hw][u * G + j];
#pragma unroll
          for (int i = 0; i < V; ++i) o[j][i] = fmaf(pu, vf[u][i], o[j][i]);
        }
      __syncwarp();
    }
    float lsum = l_own;
#pragma unroll
    for (int off = 8; off >= G; off >>= 1) lsum += __shfl_xor_sync(full, lsum, off);
    if (t < G) {
      float mt = m[0];
#pragma unroll
      for (int j = 1; j < G; ++j) mt = (j == t) ? m[j] : mt;
      sm.hm[hw][t] = mt;
      sm.hl[hw][t] = lsum;
    }
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
      for (int i = 0; i < V; ++i) sm.ho[hw][j][t * V + i] = o[j][i];
  }
  __syncthreads();
  // merge the half-warps into this CTA's partial
  for (int x = tid; x < G * D; x += kQfThreads) {
    const int j = x / D, d = x % D;
    float M = -INFINITY;
    for (int w = 0; w < 2 * kQfAttnWarps; ++w) M = fmaxf(M, sm.hm[w][j]);
    float acc = 0.f, L = 0.f;
    if (M != -INFINITY)
      for (int w = 0; w < 2 * kQfAttnWarps; ++w) {
        const float f = exp2f(sm.hm[w][j] - M);
        acc = fmaf(sm.ho[w][j][d], f, acc);
        L = fmaf(sm.hl[w][j], f, L);
      }
    sm.co[j][d] = acc;
    if (d == 0) {
      sm.cm[j] = M;
      sm.cl[j] = L;
    }
  }
  cluster.sync();                                     // every partial complete
  if (rank == 0) {
    if (tid < kQfCtas * G) {
      const QfSmem<G>* peer = cluster.map_shared_rank(&sm, tid / G);
      sm.all_m[tid] = peer->cm[tid % G];
      sm.all_l[tid] = peer->cl[tid % G];
    }
    __syncthreads();
    for (int x = tid; x < G * D; x += kQfThreads) {
      const int j = x / D, d = x % D;
      float ov[kQfCtas];
#pragma unroll
      for (int r = 0; r < kQfCtas; ++r) ov[r] = cluster.map_shared_rank(&sm, r)->co[j][d];
      float M = -INFINITY;
#pragma unroll
      for (int r = 0; r < kQfCtas; ++r) M = fmaxf(M, sm.all_m[r * G + j]);
      float acc = 0.f, L = 0.f;
      if (M != -INFINITY)
#pragma unroll
        for (int r = 0; r < kQfCtas; ++r) {
          const float f = exp2f(sm.all_m[r * G + j] - M);
          acc = fmaf(ov[r], f, acc);
          L = fmaf(sm.all_l[r * G + j], f, L);
        }
      a.o[((int64_t)b * kv.Hq + g * G + j) * D + d] = __float2bfloat16(L > 0.f ? acc / L : 0.f);
    }
  }
  cluster.sync();                                     // peers stay until CTA 0 has read them
}

template <int G>
se_status launch_fused(const QfArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(QfSmem<G>);
  static std::atomic<uint64_t> attr{0};
  if (!allow_smem(reinterpret_cast<const void*>(&quest_fused_kernel<G>), (int)smem, attr))
    return SE_ERR_CUDA;
  se_launch(quest_fused_kernel<G>, dim3(kQfCtas * a.kv.Hkv, a.kv.B), kQfThreads, smem, st, a);
  return SE_OK;
}

}  // namespace

}  // namespace se

using namespace se;

extern "C" se_status se_quest_decode_step(const se_paged_kv* kv, const void* kmin, const void* kmax,
                                          const void* q, int32_t top_pages, void* o,
                                          int32_t* page_idx, int32_t* n_sel, void* stream) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (kmin == nullptr || kmax == nullptr || q == nullptr || o == nullptr || top_pages < 0)
    return SE_ERR_INVALID_ARG;
  const int G = kv->Hq / kv->Hkv;
  if (kv->dtype != SE_BF16 || kv->D != 128 || top_pages > kQfMaxTop - 1 ||
      !(G == 1 || G == 2 || G == 4 || G == 8))
    return SE_ERR_UNSUPPORTED;
  QfArgs a{*kv, static_cast<const __nv_bfloat16*>(kmin), static_cast<const __nv_bfloat16*>(kmax),
           static_cast<const __nv_bfloat16*>(q), static_cast<__nv_bfloat16*>(o), page_idx, n_sel,
           top_pages};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (G) {
    case 1: s = launch_fused<1>(a, st); break;
    case 2: s = launch_fused<2>(a, st); break;
    case 4: s = launch_fused<4>(a, st); break;
    default: s = launch_fused<8>(a, st); break;
  }
  if (s != SE_OK) return s;
  return se_last_launch_status();
}
