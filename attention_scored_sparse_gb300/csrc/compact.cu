// Physical compaction, move-last eviction, append and prefix-span pruning.
//
// SparseEngine, "How it works": physical eviction rewrites the retained slot
// mapping and the context length and returns discarded slots to the
// allocator; the CacheManager allocates, writes, updates and frees.
// SparseEngine, "How it differs": prefix pruning R' = (R \ T) U I on idle
// blocks, logical prefix untouched.
//
// Every state change is split into a plan kernel (validation, page
// accounting, prefix sums over sequences, free-list pops into the
// workspace) and apply kernels that only run when the plan found no error,
// so a call that reports a device error leaves the cache untouched.  Fresh
// pages are popped from the top of the free-list stack in ascending
// (sequence, block) order and old pages pushed afterwards in the same order;
// the same order makes block tables and the free list deterministic.
#include "compact_ws.cuh"

namespace se {

// compact_decode_kernel's launcher (decode.cu)
se_status launch_compact_decode(const se_paged_kv* kv, const int32_t* keep, int32_t keep_stride,
                                const int32_t* first_slot, const float* aux, int64_t aux_stride,
                                const CompactWs& w, const void* q, void* o, int32_t max_entries,
                                cudaStream_t st);

// ---------------------------------------------------------------------------
// FRESH_PAGES compaction
// ---------------------------------------------------------------------------

// One CTA: validation, page counts, prefix sums, pops into the workspace.
__global__ void __launch_bounds__(1024) compact_plan_kernel(
    se_paged_kv kv, const int32_t* __restrict__ n_keep, const int32_t* __restrict__ first_slot,
    int32_t max_keep, const int32_t* __restrict__ abort_in, CompactWs w) {
  pdl_enter();
  __shared__ int tmp[33];
  __shared__ int s_bad;
  __shared__ int s_run_new;
  const int tid = threadIdx.x;
  const int P = kv.page_size;
  if (tid == 0) {
    s_bad = (abort_in != nullptr && *abort_in != 0) ? 1 : 0;
    s_run_new = 0;
  }
  __syncthreads();
  if (s_bad) {
    if (tid == 0) w.ctrl->abort = 1;
    return;
  }
  // per-sequence plan + prefix of fresh pages
  for (int b0 = 0; b0 < kv.B; b0 += blockDim.x) {
    const int b = b0 + tid;
    int nn = 0;
    if (b < kv.B) {
      const int ctx = kv.ctx_len[b];
      const int fs = first_slot[b];
      const int nk = n_keep[b];
      const bool ok = fs >= 0 && fs <= ctx && nk >= 0 && nk <= ctx - fs && nk <= max_keep &&
                      ctx <= kv.max_pages_per_seq * P;
      if (!ok) {
        set_status(kv.status, SE_ERR_BOUNDS);
        atomicExch(&s_bad, 1);
      }
      // an empty rewrite (first_slot = ctx, nothing kept) leaves the sequence as it is
      const int pb = (fs == ctx && nk == 0) ? cdiv(ctx, P) : fs / P;
      const int nctx = fs + nk;
      nn = ok ? max(cdiv(nctx, P) - pb, 0) : 0;
      w.pb[b] = pb;
      w.n_new[b] = nn;
      w.push_count[b] = 0;   // counted by the gather
      w.old_blocks[b] = cdiv(ctx, P);
      w.new_ctx[b] = nctx;
      w.old_ctx[b] = ctx;
    }
    int total;
    int ex = block_exclusive_scan(nn, tmp, &total);
    if (b < kv.B) w.off_new[b] = s_run_new + ex;
    __syncthreads();
    if (tid == 0) s_run_new += total;
    __syncthreads();
  }
  const int top0 = *kv.free_top;
  const int total_new = s_run_new;
  if (tid == 0) {
    w.ctrl->top0 = top0;
    w.ctrl->total_new = total_new;
    int bad = s_bad;
    if (!bad && total_new > top0) {
      set_status(kv.status, SE_ERR_OUT_OF_PAGES);
      bad = 1;
    }
    w.ctrl->abort = bad;
  }
}

// Copies the surviving entries into the fresh pages (K, V) and stages their
// slot_map / aux values.  grid: (entry chunks, Hkv, B).
template <int CHUNKS>  // 16-byte chunks per entry row
__global__ void __launch_bounds__(256, 8) compact_gather_kernel(
    se_paged_kv kv, const int32_t* __restrict__ keep_idx, int32_t keep_stride,
    const int32_t* __restrict__ first_slot, const float* __restrict__ aux, int64_t aux_stride,
    CompactWs w, int entries_per_cta) {
  pdl_enter();
  if (w.ctrl->abort) return;
  const int h = blockIdx.y, b = blockIdx.z;
  const int P = kv.page_size;
  const int pb = w.pb[b];
  const int fs = first_slot[b];
  const int top0 = w.ctrl->top0;
  const int pop0 = top0 - 1 - w.off_new[b];   // free_list index of this sequence's first fresh page
  if (blockIdx.x == 0 && h == 0) record_fresh_pages(kv, w, b);
  const int head = fs - pb * P;
  const int total = head + (w.new_ctx[b] - fs);
  const int e0 = blockIdx.x * entries_per_cta;
  if (e0 >= total) return;
  const int e1 = min(e0 + entries_per_cta, total);
  const int old_ctx = w.old_ctx[b];
  const int32_t* keep = keep_idx + ((int64_t)b * kv.Hkv + h) * keep_stride;
  const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
  const int esz = (int)elem_size(kv.dtype);
  const int64_t row_bytes = (int64_t)kv.D * esz;          // = CHUNKS * 16
  const int64_t page_bytes = (int64_t)kv.Hkv * P * row_bytes;
  const char* kp = static_cast<const char*>(kv.k_pool);
  const char* vp = static_cast<const char*>(kv.v_pool);
  char* kpw = static_cast<char*>(kv.k_pool);
  char* vpw = static_cast<char*>(kv.v_pool);
  constexpr int EPP = 256 / CHUNKS;  // entries per pass
  constexpr int PASSES = 2;          // entries_per_cta == EPP * PASSES
  const int sub = threadIdx.x / CHUNKS, ch = threadIdx.x % CHUNKS;
  const int64_t tmp_base = ((int64_t)b * kv.Hkv + h) * w.row;
  // all loads of this thread first (PASSES x (K, V) 16-byte rows in flight), then the stores
  uint4 kbuf[PASSES], vbuf[PASSES];
  int64_t dst[PASSES];
#pragma unroll
  for (int pss = 0; pss < PASSES; ++pss) {
    const int i = e0 + sub + pss * EPP;
    dst[pss] = -1;
    if (i >= e1) continue;
    int src;
    if (i < head) {
      src = pb * P + i;
    } else {
      src = keep[i - head];
      const bool ok = src >= fs && src < old_ctx && (i == head || src > keep[i - head - 1]);
      if (!ok) {
        if (ch == 0) {
          set_status(kv.status, SE_ERR_BOUNDS);
          atomicExch(&w.ctrl->abort, 1);
        }
        continue;
      }
    }
    const int sp = bt[src / P];
    const int dp = kv.free_list[pop0 - i / P];
    if (sp < 0 || sp >= kv.num_pages || dp < 0 || dp >= kv.num_pages) {
      if (ch == 0) {
        set_status(kv.status, SE_ERR_BOUNDS);
        atomicExch(&w.ctrl->abort, 1);
      }
      continue;
    }
    const int64_t so = (int64_t)sp * page_bytes + ((int64_t)h * P + src % P) * row_bytes + ch * 16;
    dst[pss] = (int64_t)dp * page_bytes + ((int64_t)h * P + i % P) * row_bytes + ch * 16;
    kbuf[pss] = ldg_nc_v4(kp + so);
    vbuf[pss] = ldg_nc_v4(vp + so);
    if (ch == 0) {
      w.slot_tmp[tmp_base + i] = kv.slot_map[((int64_t)b * kv.Hkv + h) *
                                                 ((int64_t)kv.max_pages_per_seq * P) + src];
      if (aux != nullptr && w.aux_tmp != nullptr)
        w.aux_tmp[tmp_base + i] = aux[((int64_t)b * kv.Hkv + h) * aux_stride + src];
    }
  }
#pragma unroll
  for (int pss = 0; pss < PASSES; ++pss) {
    if (dst[pss] < 0) continue;
    stg_v4(kpw + dst[pss], kbuf[pss]);
    stg_v4(vpw + dst[pss], vbuf[pss]);
  }
}

// Commits block tables, lengths, refcounts and free-list pushes of sequence
// b (one CTA).  Every thread takes kCommitItems consecutive blocks per round
// with all their loads in flight, so a round costs one block scan; the scan
// keeps the pushes in ascending block order.
constexpr int kCommitItems = 4;

SE_DEV void commit_pages(const se_paged_kv& kv, const CompactWs& w, int b) {
  __shared__ int tmp[33];
  __shared__ int s_off, s_total;
  const int tid = threadIdx.x;
  const int pb = w.pb[b], nn = w.n_new[b], ob = w.old_blocks[b];
  const int top0 = w.ctrl->top0, total_new = w.ctrl->total_new;
  // pushes of the sequences before b, and of all of them
  {
    int run = 0;
    for (int b0 = 0; b0 < kv.B; b0 += blockDim.x) {
      const int bb = b0 + tid;
      const int cnt = bb < kv.B ? w.push_count[bb] : 0;
      int tot;
      const int ex = block_exclusive_scan(cnt, tmp, &tot);
      if (bb == b) s_off = run + ex;
      run += tot;
    }
    if (tid == 0) s_total = run;
  }
  __syncthreads();
  const int push_base = top0 - total_new + s_off;
  const int off_new = w.off_new[b];
  int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
  const int end = max(ob, pb + nn);
  int running = 0;
  for (int c0 = pb; c0 < end; c0 += blockDim.x * kCommitItems) {
    int old[kCommitItems], np[kCommitItems], rc[kCommitItems];
#pragma unroll
    for (int i = 0; i < kCommitItems; ++i) {
      const int blk = c0 + tid * kCommitItems + i;
      old[i] = blk < ob ? bt[blk] : -1;
      np[i] = (blk < end && blk < pb + nn) ? w.newpage[off_new + blk - pb] : -1;
    }
#pragma unroll
    for (int i = 0; i < kCommitItems; ++i)
      rc[i] = (old[i] >= 0 && kv.page_refcount != nullptr) ? kv.page_refcount[old[i]] : 1;
    int n_push = 0;
#pragma unroll
    for (int i = 0; i < kCommitItems; ++i) n_push += (old[i] >= 0 && rc[i] <= 1) ? 1 : 0;
    int total;
    int pos = block_exclusive_scan(n_push, tmp, &total);
#pragma unroll
    for (int i = 0; i < kCommitItems; ++i) {
      const int blk = c0 + tid * kCommitItems + i;
      if (blk < end) {
        bt[blk] = np[i];
        if (np[i] >= 0 && kv.page_refcount) kv.page_refcount[np[i]] = 1;
      }
      if (old[i] >= 0) {
        if (rc[i] <= 1) {
          if (push_base + running + pos < kv.num_pages) {
            kv.free_list[push_base + running + pos] = old[i];
            if (kv.page_refcount) kv.page_refcount[old[i]] = 0;
          }
          ++pos;
        } else {
          atomicSub(&kv.page_refcount[old[i]], 1);
        }
      }
    }
    running += total;
  }
  if (tid == 0) {
    kv.ctx_len[b] = w.new_ctx[b];
    if (b == 0) *kv.free_top = top0 - total_new + s_total;
  }
}

// Commits slot maps (and aux) of (b, h), slots [chunk * 4096, +4096) from
// the rewritten base, from the staged values; slots past the new length
// become -1 (aux 0).
SE_DEV void commit_slots(const se_paged_kv& kv, float* aux, int64_t aux_stride,
                         const CompactWs& w, int b, int h, int chunk) {
  const int P = kv.page_size;
  const int base = w.pb[b] * P;
  const int nctx = w.new_ctx[b], octx = w.old_ctx[b];
  const int s_end = max(nctx, octx);
  const int s0 = base + chunk * 4096;
  if (s0 >= s_end) return;
  const int s1 = min(s0 + 4096, s_end);
  const int64_t smax = (int64_t)kv.max_pages_per_seq * P;
  int32_t* sm = kv.slot_map + ((int64_t)b * kv.Hkv + h) * smax;
  const int64_t tb = ((int64_t)b * kv.Hkv + h) * w.row;
  float* ar = aux != nullptr ? aux + ((int64_t)b * kv.Hkv + h) * aux_stride : nullptr;
  for (int s = s0 + threadIdx.x; s < s1; s += blockDim.x) {
    if (s < nctx) {
      sm[s] = w.slot_tmp[tb + (s - base)];
      if (ar) ar[s] = w.aux_tmp[tb + (s - base)];
    } else {
      sm[s] = -1;
      if (ar) ar[s] = 0.f;
    }
  }
}

// Commit of a compaction.  grid: (1 + slot chunks of 4096, Hkv, B), 1024
// threads; CTA (0, 0, b) commits the pages of sequence b, CTA (1 + c, h, b)
// chunk c of the slot map of (b, h).  Nothing runs after a planning error.
__global__ void __launch_bounds__(1024, 2) compact_commit_kernel(se_paged_kv kv, float* aux,
                                                              int64_t aux_stride, CompactWs w) {
  pdl_enter();
  if (w.ctrl->abort) return;
  const int h = blockIdx.y, b = blockIdx.z;
  if (blockIdx.x == 0) {
    if (h == 0) commit_pages(kv, w, b);
    return;
  }
  commit_slots(kv, aux, aux_stride, w, b, h, blockIdx.x - 1);
}

// ---------------------------------------------------------------------------
// MOVE_LAST eviction (H2O)
// ---------------------------------------------------------------------------

struct MoveWs {
  CompactCtrl* ctrl;
};

static MoveWs carve_move(const se_paged_kv* kv, void* ws, size_t* bytes) {
  WsCarver c(ws);
  MoveWs w;
  w.ctrl = c.take<CompactCtrl>(1);
  *bytes = c.bytes();
  return w;
}

// Move-last eviction in one launch.  grid: B, 256 threads (one warp per KV
// head).  Every CTA validates the victims of every sequence (all heads evict
// or none) and takes the free-list rank of its sequence's emptied page from a
// scan over the sequences before it; a call with an invalid sequence changes
// nothing.  CTA b moves the last entry of sequence b into each head's victim
// slot and pushes the page the move empties; the last CTA to finish commits
// the lengths and the free-list top, which every CTA read first.
__global__ void __launch_bounds__(256) move_last_kernel(se_paged_kv kv,
                                                        const int32_t* __restrict__ victim,
                                                        float* aux, int64_t aux_stride, MoveWs w) {
  pdl_enter();
  __shared__ int tmp[33];
  __shared__ int s_bad, s_off, s_act;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int P = kv.page_size;
  const int top0 = *kv.free_top;
  if (tid == 0) {
    s_bad = 0;
    s_off = 0;
    s_act = 0;
  }
  __syncthreads();
  int run = 0;   // pages pushed by the sequences before the current chunk
  for (int b0 = 0; b0 < kv.B; b0 += blockDim.x) {
    const int bb = b0 + tid;
    int freed = 0;
    if (bb < kv.B) {
      const int ctx = kv.ctx_len[bb];
      int n_neg = 0, n_ok = 0;
      for (int h = 0; h < kv.Hkv; ++h) {
        const int v = victim[bb * kv.Hkv + h];
        n_neg += v < 0;
        n_ok += (v >= 0 && v < ctx);
      }
      if (n_neg != kv.Hkv && n_ok != kv.Hkv) {
        set_status(kv.status, n_neg > 0 ? SE_ERR_UNEVEN : SE_ERR_BOUNDS);
        atomicExch(&s_bad, 1);
      }
      freed = (n_ok == kv.Hkv && (ctx - 1) % P == 0) ? 1 : 0;
      if (bb == b) s_act = n_ok == kv.Hkv ? 1 : 0;
    }
    int total;
    const int ex = block_exclusive_scan(freed, tmp, &total);
    if (bb == b) s_off = run + ex;
    run += total;
  }
  __syncthreads();
  const bool bad = s_bad != 0;
  if (!bad && s_act) {
    const int last = kv.ctx_len[b] - 1;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int esz = (int)elem_size(kv.dtype);
    const int64_t row_bytes = (int64_t)kv.D * esz;
    const int chunks = (int)(row_bytes / 16);
    const int64_t page_bytes = (int64_t)kv.Hkv * P * row_bytes;
    const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
    const int64_t smax = (int64_t)kv.max_pages_per_seq * P;
    for (int h = warp; h < kv.Hkv; h += blockDim.x >> 5) {
      const int v = victim[b * kv.Hkv + h];
      if (v != last) {
        const int64_t so = (int64_t)bt[last / P] * page_bytes + ((int64_t)h * P + last % P) * row_bytes;
        const int64_t dof = (int64_t)bt[v / P] * page_bytes + ((int64_t)h * P + v % P) * row_bytes;
        for (int c = lane; c < chunks; c += 32) {
          const uint4 k4 = ldg_v4(static_cast<const char*>(kv.k_pool) + so + c * 16);
          const uint4 v4 = ldg_v4(static_cast<const char*>(kv.v_pool) + so + c * 16);
          stg_v4(static_cast<char*>(kv.k_pool) + dof + c * 16, k4);
          stg_v4(static_cast<char*>(kv.v_pool) + dof + c * 16, v4);
        }
      }
      if (lane == 0) {
        int32_t* sm = kv.slot_map + ((int64_t)b * kv.Hkv + h) * smax;
        const int pos = sm[last];
        sm[v] = pos;
        sm[last] = -1;
        if (aux != nullptr) {
          float* ar = aux + ((int64_t)b * kv.Hkv + h) * aux_stride;
          const float a = ar[last];
          ar[v] = a;
          ar[last] = 0.f;
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == 0 && last % P == 0) {
      const int page = bt[last / P];
      kv.block_table[(int64_t)b * kv.max_pages_per_seq + last / P] = -1;
      if (kv.page_refcount) kv.page_refcount[page] = 0;
      kv.free_list[top0 + s_off] = page;
    }
  }
  if (finish_cta(&w.ctrl->done) && !bad) {
    for (int bb = tid; bb < kv.B; bb += blockDim.x) {
      const int ctx = kv.ctx_len[bb];
      int n_ok = 0;
      for (int h = 0; h < kv.Hkv; ++h) {
        const int v = victim[bb * kv.Hkv + h];
        n_ok += (v >= 0 && v < ctx);
      }
      if (n_ok == kv.Hkv) kv.ctx_len[bb] = ctx - 1;
    }
    if (tid == 0) *kv.free_top = top0 + run;
  }
}

// ---------------------------------------------------------------------------
// Append (CacheManager write)
// ---------------------------------------------------------------------------

struct AppendWs {
  CompactCtrl* ctrl;
};

static AppendWs carve_append(const se_paged_kv* kv, void* ws, size_t* bytes) {
  WsCarver c(ws);
  AppendWs w;
  w.ctrl = c.take<CompactCtrl>(1);
  *bytes = c.bytes();
  return w;
}

// Block blockIdx.x of the append of sequence b (see append_kernel); base:
// pop rank of the sequence's first fresh page, top0: the free-list top
// before the call.
SE_DEV void append_fill_body(se_paged_kv kv, const void* __restrict__ k_new,
                             const void* __restrict__ v_new, int n, float* aux, int64_t aux_stride,
                             void* kmin, void* kmax, int b, int base, int top0) {
  const int P = kv.page_size;
  const int ctx = kv.ctx_len[b];
  const int logical = kv.logical_len[b];
  const int blk = ctx / P + blockIdx.x;
  const int s0 = max(ctx, blk * P), s1 = min(ctx + n, (blk + 1) * P);   // slots filled here
  const int64_t mps = kv.max_pages_per_seq;
  if (s0 < s1) {
    const bool fresh = blk * P >= ctx;   // the block held nothing before
    const int page = fresh ? kv.free_list[top0 - 1 - (base + blk - cdiv(ctx, P))]
                           : kv.block_table[b * mps + blk];
    const int esz = (int)elem_size(kv.dtype);
    const int64_t row_bytes = (int64_t)kv.D * esz;
    const int chunks = (int)(row_bytes / 16);
    const int64_t page_bytes = (int64_t)kv.Hkv * P * row_bytes;
    const int rows = (s1 - s0) * kv.Hkv;
    for (int t = threadIdx.x; t < rows * chunks; t += blockDim.x) {
      const int r = t / chunks, c = t % chunks;
      const int slot = s0 + r / kv.Hkv, h = r % kv.Hkv;
      const int64_t so = (((int64_t)b * n + (slot - ctx)) * kv.Hkv + h) * row_bytes + c * 16;
      const int64_t dof = (int64_t)page * page_bytes + ((int64_t)h * P + slot % P) * row_bytes + c * 16;
      stg_v4(static_cast<char*>(kv.k_pool) + dof, ldg_v4(static_cast<const char*>(k_new) + so));
      stg_v4(static_cast<char*>(kv.v_pool) + dof, ldg_v4(static_cast<const char*>(v_new) + so));
    }
    if (kmin != nullptr) {
      // Quest bounds: a fresh page starts from its first key, an old page widens
      for (int x = threadIdx.x; x < kv.Hkv * kv.D; x += blockDim.x) {
        const int h = x / kv.D, d = x % kv.D;
        const int64_t mo = ((int64_t)page * kv.Hkv + h) * kv.D + d;
        if (kv.dtype == SE_BF16) {
          const __nv_bfloat16* kn = static_cast<const __nv_bfloat16*>(k_new);
          __nv_bfloat16* mn = static_cast<__nv_bfloat16*>(kmin) + mo;
          __nv_bfloat16* mx = static_cast<__nv_bfloat16*>(kmax) + mo;
          __nv_bfloat16 lo = fresh ? kn[(((int64_t)b * n + (s0 - ctx)) * kv.Hkv + h) * kv.D + d] : *mn;
          __nv_bfloat16 hi = fresh ? lo : *mx;
          for (int slot = s0; slot < s1; ++slot) {
            const __nv_bfloat16 k = kn[(((int64_t)b * n + (slot - ctx)) * kv.Hkv + h) * kv.D + d];
            if (__bfloat162float(k) < __bfloat162float(lo)) lo = k;
            if (__bfloat162float(k) > __bfloat162float(hi)) hi = k;
          }
          *mn = lo;
          *mx = hi;
        } else {
          const float* kn = static_cast<const float*>(k_new);
          float* mn = static_cast<float*>(kmin) + mo;
          float* mx = static_cast<float*>(kmax) + mo;
          float lo = fresh ? INFINITY : *mn, hi = fresh ? -INFINITY : *mx;
          for (int slot = s0; slot < s1; ++slot) {
            const float k = kn[(((int64_t)b * n + (slot - ctx)) * kv.Hkv + h) * kv.D + d];
            lo = fminf(lo, k);
            hi = fmaxf(hi, k);
          }
          *mn = lo;
          *mx = hi;
        }
      }
    }
    const int64_t smax = mps * P;
    for (int x = threadIdx.x; x < (s1 - s0) * kv.Hkv; x += blockDim.x) {
      const int slot = s0 + x / kv.Hkv, h = x % kv.Hkv;
      kv.slot_map[((int64_t)b * kv.Hkv + h) * smax + slot] = logical + (slot - ctx);
      if (aux != nullptr) aux[((int64_t)b * kv.Hkv + h) * aux_stride + slot] = 0.f;
    }
    if (threadIdx.x == 0 && fresh) {
      kv.block_table[b * mps + blk] = page;
      if (kv.page_refcount) kv.page_refcount[page] = 1;
    }
  }

}

// Append in one launch.  grid: (cdiv(n + P - 1, P), B), 256 threads.  Every
// CTA checks the bounds of every sequence and the free-list capacity and
// takes its sequence's pop rank (fresh pages in ascending (b, block) order)
// from a scan over the sequences; a call that fails a check changes nothing.
// CTA (j, b) fills block ctx / P + j of sequence b: K/V rows, slot map, aux,
// Quest bounds, and the block-table entry of a fresh page.  The last CTA to
// finish commits both lengths of every sequence and the free-list top, which
// every CTA read first.
__global__ void __launch_bounds__(256) append_kernel(se_paged_kv kv,
                                                     const void* __restrict__ k_new,
                                                     const void* __restrict__ v_new, int n,
                                                     float* aux, int64_t aux_stride,
                                                     void* kmin, void* kmax, AppendWs w) {
  pdl_enter();
  __shared__ int tmp[33];
  __shared__ int s_bad, s_base;
  const int b = blockIdx.y, tid = threadIdx.x;
  const int P = kv.page_size;
  const int top0 = *kv.free_top;
  if (tid == 0) {
    s_bad = 0;
    s_base = 0;
  }
  __syncthreads();
  int run = 0;   // fresh pages of the sequences before the current chunk
  for (int b0 = 0; b0 < kv.B; b0 += blockDim.x) {
    const int bb = b0 + tid;
    int need = 0;
    if (bb < kv.B) {
      const int c = kv.ctx_len[bb];
      if (c < 0 || (int64_t)c + n > (int64_t)kv.max_pages_per_seq * P) {
        set_status(kv.status, SE_ERR_BOUNDS);
        atomicExch(&s_bad, 1);
      } else {
        need = cdiv(c + n, P) - cdiv(c, P);
      }
    }
    int total;
    const int ex = block_exclusive_scan(need, tmp, &total);
    if (bb == b) s_base = run + ex;
    run += total;
  }
  __syncthreads();
  bool bad = s_bad != 0;
  if (!bad && run > top0) {
    if (tid == 0) set_status(kv.status, SE_ERR_OUT_OF_PAGES);
    bad = true;
  }
  if (!bad) append_fill_body(kv, k_new, v_new, n, aux, aux_stride, kmin, kmax, b, s_base, top0);
  if (finish_cta(&w.ctrl->done) && !bad) {
    for (int bb = tid; bb < kv.B; bb += blockDim.x) {
      kv.ctx_len[bb] += n;
      kv.logical_len[bb] += n;
    }
    if (tid == 0) *kv.free_top = top0 - run;
  }
}


// ---------------------------------------------------------------------------
// Prefix-span pruning plan
// ---------------------------------------------------------------------------

struct PruneWs {
  int32_t* abort;    // [1]
  int32_t* keep;     // [B][Hkv][smax]
  int32_t* n_keep;   // [B]
  int32_t* first;    // [B]
  void* compact_ws;
  size_t compact_bytes;
};

static PruneWs carve_prune(const se_paged_kv* kv, void* ws, size_t* bytes) {
  WsCarver c(ws);
  PruneWs w;
  const int64_t smax = (int64_t)kv->max_pages_per_seq * kv->page_size;
  w.abort = c.take<int32_t>(1);
  w.keep = c.take<int32_t>((size_t)kv->B * kv->Hkv * smax);
  w.n_keep = c.take<int32_t>(kv->B);
  w.first = c.take<int32_t>(kv->B);
  size_t cb = 0;
  carve_compact(kv, (int32_t)smax, nullptr, true, &cb);
  char* cws = c.take<char>(cb);
  w.compact_ws = cws;
  w.compact_bytes = cb;
  *bytes = c.bytes();
  return w;
}

// Slots per thread and round of the prune plan's keep-list scan.
constexpr int kPruneItems = 4;

// grid: B, 1024 threads.  Builds per-head keep lists for R' = (R \ T) U I.
// The first rewritten slot is the lowest slot of any head whose position is
// at least L: each thread stops at its first such slot of a head (its slots
// are visited in increasing order) and the warps meet in one shared minimum.
// The keep lists come from one block scan per kPruneItems x 1024 slots, each
// thread taking kPruneItems consecutive slots in order.
__global__ void __launch_bounds__(1024) prune_plan_kernel(se_paged_kv kv,
                                                          const int32_t* __restrict__ Lp,
                                                          const int32_t* __restrict__ Rp,
                                                          const uint8_t* __restrict__ mask,
                                                          int32_t mask_stride, int32_t* n_busy,
                                                          PruneWs w) {
  pdl_enter();
  __shared__ int tmp[33];
  __shared__ int s_first, s_busy, s_count0, s_bad;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int P = kv.page_size;
  const int ctx = kv.ctx_len[b];
  const int L = Lp[b], R = Rp[b];
  const int64_t smax = (int64_t)kv.max_pages_per_seq * P;
  if (tid == 0) { s_first = ctx; s_busy = 0; s_count0 = -1; s_bad = 0; }
  __syncthreads();
  {
    int first = ctx;
    for (int h = 0; h < kv.Hkv; ++h) {
      const int32_t* sm = kv.slot_map + ((int64_t)b * kv.Hkv + h) * smax;
      for (int s = tid; s < min(ctx, first); s += blockDim.x)
        if (sm[s] >= L) {
          first = s;
          break;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
    if ((tid & 31) == 0 && first < ctx) atomicMin(&s_first, first);
  }
  __syncthreads();
  const int fs = s_first;
  const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
  if (kv.page_refcount != nullptr) {
    int cnt = 0;
    for (int blk = fs / P + tid; blk < cdiv(ctx, P); blk += blockDim.x)
      cnt += kv.page_refcount[bt[blk]] > 1;
    if (cnt) atomicAdd(&s_busy, cnt);
  }
  for (int h = 0; h < kv.Hkv; ++h) {
    const int32_t* sm = kv.slot_map + ((int64_t)b * kv.Hkv + h) * smax;
    int32_t* keep = w.keep + ((int64_t)b * kv.Hkv + h) * smax;
    int running = 0;
    for (int c0 = fs; c0 < ctx; c0 += blockDim.x * kPruneItems) {
      const int s0 = c0 + tid * kPruneItems;
      int pos[kPruneItems];
#pragma unroll
      for (int i = 0; i < kPruneItems; ++i) pos[i] = s0 + i < ctx ? sm[s0 + i] : -1;
      bool k[kPruneItems];
      int n = 0;
#pragma unroll
      for (int i = 0; i < kPruneItems; ++i) {
        const int s = s0 + i;
        bool leaves = false;
        if (s < ctx && pos[i] >= L && pos[i] < R) {
          if (pos[i] - L >= mask_stride) {
            set_status(kv.status, SE_ERR_BOUNDS);
            atomicExch(w.abort, 1);
          }
          const bool in_I =
              pos[i] - L < mask_stride && mask[(int64_t)b * mask_stride + (pos[i] - L)] != 0;
          const bool busy = kv.page_refcount != nullptr && kv.page_refcount[bt[s / P]] > 1;
          leaves = !in_I && !busy;
        }
        k[i] = s < ctx && !leaves;
        n += k[i] ? 1 : 0;
      }
      int total;
      int at = running + block_exclusive_scan(n, tmp, &total);
#pragma unroll
      for (int i = 0; i < kPruneItems; ++i)
        if (k[i]) keep[at++] = s0 + i;
      running += total;
    }
    if (tid == 0) {
      if (h == 0) s_count0 = running;
      else if (running != s_count0) s_bad = 1;
    }
    __syncthreads();
  }
  if (tid == 0) {
    w.first[b] = fs;
    w.n_keep[b] = s_count0 < 0 ? 0 : s_count0;
    if (n_busy) n_busy[b] = s_busy;
    if (s_bad) {
      set_status(kv.status, SE_ERR_UNEVEN);
      atomicExch(w.abort, 1);
    }
  }
}

__global__ void zero_int_kernel(int32_t* p) {
  pdl_enter();
  *p = 0;
}

// ---------------------------------------------------------------------------
// Release of whole sequences (reclaim of an idle chain's row)
// ---------------------------------------------------------------------------

struct ReleaseWs {
  CompactCtrl* ctrl;   // abort, top0
  int32_t* count;      // [B] pages each released sequence pushes
};

static ReleaseWs carve_release(const se_paged_kv* kv, void* ws, size_t* bytes) {
  WsCarver c(ws);
  ReleaseWs w;
  w.ctrl = c.take<CompactCtrl>(1);
  w.count = c.take<int32_t>(kv->B);
  *bytes = c.bytes();
  return w;
}

SE_DEV bool release_pushes(const se_paged_kv& kv, int page) {
  return page >= 0 && (kv.page_refcount == nullptr || kv.page_refcount[page] <= 1);
}

// grid: B, 1024 threads.  Counts the pages each released sequence pushes and
// checks every page id before anything is written.  ctrl was zeroed.
__global__ void __launch_bounds__(1024) release_count_kernel(se_paged_kv kv,
                                                             const int32_t* __restrict__ mask,
                                                             ReleaseWs w) {
  pdl_enter();
  __shared__ int s_cnt;
  const int b = blockIdx.x;
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  if (b == 0 && threadIdx.x == 0) w.ctrl->top0 = *kv.free_top;
  int cnt = 0;
  if (mask[b] != 0) {
    const int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
    for (int blk = threadIdx.x; blk < kv.max_pages_per_seq; blk += blockDim.x) {
      const int page = bt[blk];
      if (page >= kv.num_pages) {
        set_status(kv.status, SE_ERR_BOUNDS);
        atomicExch(&w.ctrl->abort, 1);
      } else if (release_pushes(kv, page)) {
        cnt++;
      }
    }
  }
  if (cnt) atomicAdd(&s_cnt, cnt);
  __syncthreads();
  if (threadIdx.x == 0) w.count[b] = s_cnt;
}

// grid: B, 1024 threads.  Pushes (ascending sequence, then block), drops the
// references of shared pages, clears block table, slot map and lengths.
__global__ void __launch_bounds__(1024) release_apply_kernel(se_paged_kv kv,
                                                             const int32_t* __restrict__ mask,
                                                             ReleaseWs w) {
  pdl_enter();
  __shared__ int tmp[33];
  __shared__ int s_off, s_total;
  if (w.ctrl->abort) return;
  const int b = blockIdx.x, tid = threadIdx.x;
  if (tid == 0) {
    int off = 0, total = 0;
    for (int bb = 0; bb < kv.B; ++bb) {
      off += bb < b ? w.count[bb] : 0;
      total += w.count[bb];
    }
    s_off = off;
    s_total = total;
  }
  __syncthreads();
  const int top0 = w.ctrl->top0;
  if (b == 0 && tid == 0) {
    if (top0 + s_total > kv.num_pages) set_status(kv.status, SE_ERR_BOUNDS);
    else *kv.free_top = top0 + s_total;
  }
  if (mask[b] == 0 || top0 + s_total > kv.num_pages) return;
  int32_t* bt = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
  int running = 0;
  for (int c0 = 0; c0 < kv.max_pages_per_seq; c0 += blockDim.x) {
    const int blk = c0 + tid;
    const int page = blk < kv.max_pages_per_seq ? bt[blk] : -1;
    const bool push = release_pushes(kv, page);
    int total;
    const int pos = block_exclusive_scan(push ? 1 : 0, tmp, &total);
    if (push) {
      kv.free_list[top0 + s_off + running + pos] = page;
      if (kv.page_refcount) kv.page_refcount[page] = 0;
    } else if (page >= 0) {
      atomicSub(&kv.page_refcount[page], 1);   // shared: this sequence's reference only
    }
    if (blk < kv.max_pages_per_seq) bt[blk] = -1;
    running += total;
  }
  const int64_t smax = (int64_t)kv.max_pages_per_seq * kv.page_size;
  int32_t* sm = kv.slot_map + (int64_t)b * kv.Hkv * smax;
  for (int64_t x = tid; x < kv.Hkv * smax; x += blockDim.x) sm[x] = -1;
  if (tid == 0) {
    kv.ctx_len[b] = 0;
    kv.logical_len[b] = 0;
  }
}


}  // namespace se

using namespace se;

// ---------------------------------------------------------------------------
// Host entry points
// ---------------------------------------------------------------------------

static se_status launch_compact_gather(const se_paged_kv* kv, const int32_t* keep_idx,
                                       int32_t keep_stride, const int32_t* first_slot,
                                       int32_t max_keep, float* aux, int64_t aux_stride,
                                       const CompactWs& w, cudaStream_t st) {
  const int row_bytes = kv->D * (int)elem_size(kv->dtype);
  const int chunks = row_bytes / 16;
  const int max_entries = max_keep + kv->page_size;
  // entries per CTA = (256 / chunks) rows per pass x 2 passes (more, smaller CTAs measured
  // faster than 4 or 8 passes for both the SnapKV compaction and the Kara prune)
  switch (chunks) {
    case 8: {
      const int epc = 2 * (256 / 8);
      se_launch(compact_gather_kernel<8>, dim3(cdiv(max_entries, epc), kv->Hkv, kv->B), 256, 0, st,
          *kv, keep_idx, keep_stride, first_slot, aux, aux_stride, w, epc);
      return SE_OK;
    }
    case 16: {
      const int epc = 2 * (256 / 16);
      se_launch(compact_gather_kernel<16>, dim3(cdiv(max_entries, epc), kv->Hkv, kv->B), 256, 0, st,
          *kv, keep_idx, keep_stride, first_slot, aux, aux_stride, w, epc);
      return SE_OK;
    }
    case 32: {
      const int epc = 2 * (256 / 32);
      se_launch(compact_gather_kernel<32>, dim3(cdiv(max_entries, epc), kv->Hkv, kv->B), 256, 0, st,
          *kv, keep_idx, keep_stride, first_slot, aux, aux_stride, w, epc);
      return SE_OK;
    }
    default:
      return SE_ERR_UNSUPPORTED;
  }
}

static void launch_compact_commit(const se_paged_kv* kv, float* aux, int64_t aux_stride,
                                  const CompactWs& w, cudaStream_t st) {
  const int max_span = kv->max_pages_per_seq * kv->page_size;
  se_launch(compact_commit_kernel, dim3(1 + cdiv(max_span, 4096), kv->Hkv, kv->B), 1024, 0, st,
      *kv, aux, aux_stride, w);
}

static se_status launch_compact(const se_paged_kv* kv, const int32_t* keep_idx,
                                int32_t keep_stride, const int32_t* n_keep,
                                const int32_t* first_slot, int32_t max_keep, float* aux,
                                int64_t aux_stride, void* ws, size_t ws_bytes,
                                const int32_t* abort_in, cudaStream_t st) {
  size_t need = 0;
  CompactWs w = carve_compact(kv, max_keep, ws, aux != nullptr, &need);
  if (ws == nullptr || ws_bytes < need) return SE_ERR_INVALID_ARG;
  const int chunks = kv->D * (int)elem_size(kv->dtype) / 16;
  if (chunks != 8 && chunks != 16 && chunks != 32) return SE_ERR_UNSUPPORTED;
  se_launch(compact_plan_kernel, 1, 1024, 0, st, *kv, n_keep, first_slot, max_keep, abort_in, w);
  se_status s = launch_compact_gather(kv, keep_idx, keep_stride, first_slot, max_keep, aux,
                                      aux_stride, w, st);
  if (s != SE_OK) return s;
  launch_compact_commit(kv, aux, aux_stride, w, st);
  return se_last_launch_status();
}

extern "C" size_t se_compact_evict_workspace_size(const se_paged_kv* kv, int32_t max_keep) {
  if (kv == nullptr) return 0;
  size_t a = 0, b = 0;
  carve_compact(kv, max_keep, nullptr, true, &a);
  carve_move(kv, nullptr, &b);
  return a > b ? a : b;
}

extern "C" se_status se_compact_evict(const se_paged_kv* kv, int32_t mode,
                                      const int32_t* keep_idx, int32_t keep_stride,
                                      const int32_t* n_keep, const int32_t* first_slot,
                                      int32_t max_keep, float* aux, int64_t aux_stride,
                                      void* workspace, size_t workspace_bytes, void* stream) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (keep_idx == nullptr || workspace == nullptr) return SE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (mode == SE_COMPACT_FRESH_PAGES) {
    if (n_keep == nullptr || first_slot == nullptr || max_keep < 0 || keep_stride < max_keep)
      return SE_ERR_INVALID_ARG;
    return launch_compact(kv, keep_idx, keep_stride, n_keep, first_slot, max_keep, aux,
                          aux_stride, workspace, workspace_bytes, nullptr, st);
  }
  if (mode == SE_COMPACT_MOVE_LAST) {
    size_t need = 0;
    MoveWs w = carve_move(kv, workspace, &need);
    if (workspace_bytes < need) return SE_ERR_INVALID_ARG;
    se_launch(move_last_kernel, kv->B, 256, 0, st, *kv, keep_idx, aux, aux_stride, w);
    return se_last_launch_status();
  }
  return SE_ERR_INVALID_ARG;
}

// Compaction and decode attention in one pass over the kept entries: the
// compaction's plan, then compact_decode_kernel (gather + decode), then its
// commit; shapes that kernel does not take run the plain compaction and then
// decode attention over the dense view of the result.
extern "C" size_t se_compact_decode_workspace_size(const se_paged_kv* kv, int32_t max_keep,
                                                   int32_t max_entries) {
  if (kv == nullptr || max_keep < 0 || max_entries < 1) return 0;
  size_t a = 0;
  carve_compact(kv, max_keep, nullptr, true, &a);
  return align_up(a, 256) + se_sparse_decode_attn_workspace_size(kv, max_entries);
}

extern "C" se_status se_compact_decode(const se_paged_kv* kv, const int32_t* keep_idx,
                                       int32_t keep_stride, const int32_t* n_keep,
                                       const int32_t* first_slot, int32_t max_keep, float* aux,
                                       int64_t aux_stride, const void* q, void* o,
                                       int32_t max_entries, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (keep_idx == nullptr || n_keep == nullptr || first_slot == nullptr || q == nullptr ||
      o == nullptr || workspace == nullptr || max_keep < 0 || keep_stride < max_keep ||
      max_entries < 1)
    return SE_ERR_INVALID_ARG;
  if (workspace_bytes < se_compact_decode_workspace_size(kv, max_keep, max_entries))
    return SE_ERR_INVALID_ARG;
  const int chunks = kv->D * (int)elem_size(kv->dtype) / 16;
  if (chunks != 8 && chunks != 16 && chunks != 32) return SE_ERR_UNSUPPORTED;
  size_t ca = 0;
  CompactWs w = carve_compact(kv, max_keep, workspace, aux != nullptr, &ca);
  ca = align_up(ca, 256);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  se_launch(compact_plan_kernel, 1, 1024, 0, st, *kv, n_keep, first_slot, max_keep,
            (const int32_t*)nullptr, w);
  s = launch_compact_decode(kv, keep_idx, keep_stride, first_slot, aux, aux_stride, w, q, o,
                            max_entries, st);
  if (s == SE_OK) {
    launch_compact_commit(kv, aux, aux_stride, w, st);
    return se_last_launch_status();
  }
  if (s != SE_ERR_UNSUPPORTED) return s;
  s = launch_compact_gather(kv, keep_idx, keep_stride, first_slot, max_keep, aux, aux_stride, w, st);
  if (s != SE_OK) return s;
  launch_compact_commit(kv, aux, aux_stride, w, st);
  s = se_last_launch_status();
  if (s != SE_OK) return s;
  return se_sparse_decode_attn(kv, q, SE_VIEW_DENSE, nullptr, 0, 0, max_entries, o, nullptr, 0,
                               static_cast<char*>(workspace) + ca, workspace_bytes - ca, stream);
}

extern "C" size_t se_append_kv_workspace_size(const se_paged_kv* kv) {
  if (kv == nullptr) return 0;
  size_t b = 0;
  carve_append(kv, nullptr, &b);
  return b;
}

extern "C" se_status se_append_kv(const se_paged_kv* kv, const void* k_new, const void* v_new,
                                  int32_t n_new, float* aux, int64_t aux_stride, void* kmin,
                                  void* kmax, void* workspace, size_t workspace_bytes,
                                  void* stream) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (k_new == nullptr || v_new == nullptr || workspace == nullptr || n_new < 0)
    return SE_ERR_INVALID_ARG;
  if ((kmin == nullptr) != (kmax == nullptr)) return SE_ERR_INVALID_ARG;
  if ((int64_t)n_new > (int64_t)kv->max_pages_per_seq * kv->page_size) return SE_ERR_INVALID_ARG;
  size_t need = 0;
  AppendWs w = carve_append(kv, workspace, &need);
  if (workspace_bytes < need) return SE_ERR_INVALID_ARG;
  if (n_new == 0) return SE_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 grid(cdiv(n_new + kv->page_size - 1, kv->page_size), kv->B);
  se_launch(append_kernel, grid, 256, 0, st, *kv, k_new, v_new, n_new, aux, aux_stride, kmin, kmax,
            w);
  return se_last_launch_status();
}

extern "C" size_t se_prune_span_workspace_size(const se_paged_kv* kv) {
  if (kv == nullptr) return 0;
  size_t b = 0;
  carve_prune(kv, nullptr, &b);
  return b;
}

extern "C" se_status se_prune_span(const se_paged_kv* kv, const int32_t* L, const int32_t* R,
                                   const uint8_t* mask, int32_t mask_stride, int32_t* n_busy,
                                   float* aux, int64_t aux_stride, void* workspace,
                                   size_t workspace_bytes, void* stream) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (L == nullptr || R == nullptr || mask == nullptr || workspace == nullptr || mask_stride < 0)
    return SE_ERR_INVALID_ARG;
  size_t need = 0;
  PruneWs w = carve_prune(kv, workspace, &need);
  if (workspace_bytes < need) return SE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int32_t smax = kv->max_pages_per_seq * kv->page_size;
  se_launch(zero_int_kernel, 1, 1, 0, st, w.abort);
  se_launch(prune_plan_kernel, kv->B, 1024, 0, st, *kv, L, R, mask, mask_stride, n_busy, w);
  return launch_compact(kv, w.keep, smax, w.n_keep, w.first, smax, aux, aux_stride, w.compact_ws,
                        w.compact_bytes, w.abort, st);
}

extern "C" size_t se_release_seqs_workspace_size(const se_paged_kv* kv) {
  if (kv == nullptr) return 0;
  size_t b = 0;
  carve_release(kv, nullptr, &b);
  return b;
}

extern "C" se_status se_release_seqs(const se_paged_kv* kv, const int32_t* mask, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  se_status s = se_check_kv(kv);
  if (s != SE_OK) return s;
  if (mask == nullptr || workspace == nullptr) return SE_ERR_INVALID_ARG;
  size_t need = 0;
  ReleaseWs w = carve_release(kv, workspace, &need);
  if (workspace_bytes < need) return SE_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(w.ctrl, 0, sizeof(CompactCtrl), st) != cudaSuccess) return SE_ERR_CUDA;
  se_launch(release_count_kernel, kv->B, 1024, 0, st, *kv, mask, w);
  se_launch(release_apply_kernel, kv->B, 1024, 0, st, *kv, mask, w);
  return se_last_launch_status();
}
