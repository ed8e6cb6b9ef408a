// Workspace of a compaction into fresh pages, shared by the plan, gather,
// commit and compaction-plus-decode kernels.
#pragma once

#include "se_common.cuh"

namespace se {

struct CompactCtrl {
  int32_t abort;
  int32_t top0;
  int32_t total_new;
  int32_t total_push;
  int32_t done;        // CTAs finished (finish_cta); zero between calls
};

// Counts the calling CTA as finished -- after a barrier over its threads and
// a device-scope fence, so that every read and write of the CTA precedes the
// count -- and returns, in every thread, whether it was the last CTA of the
// grid.  The last one resets the counter for the next call.  No CTA waits
// for another.
SE_DEV bool finish_cta(int32_t* done) {
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int n = (int)(gridDim.x * gridDim.y * gridDim.z);
    const bool last = atomicAdd(done, 1) == n - 1;
    if (last) {
      __threadfence();
      *done = 0;
    }
    s_last = last ? 1 : 0;
  }
  __syncthreads();
  return s_last != 0;
}

struct CompactWs {
  CompactCtrl* ctrl;
  int32_t* pb;        // [B] first rewritten block
  int32_t* n_new;     // [B] fresh pages
  int32_t* old_blocks;// [B] blocks before the call
  int32_t* new_ctx;   // [B]
  int32_t* old_ctx;   // [B]
  int32_t* off_new;   // [B] prefix of n_new
  int32_t* push_count;// [B] old pages of the sequence that go back to the free list
  int32_t* newpage;   // [B * max_pages_per_seq]
  int32_t* slot_tmp;  // [B][Hkv][row]  new slot_map values from pb*P on
  float* aux_tmp;     // [B][Hkv][row]
  int64_t row;        // max_keep + page_size
};

static CompactWs carve_compact(const se_paged_kv* kv, int32_t max_keep, void* ws, bool aux,
                               size_t* bytes) {
  WsCarver c(ws);
  CompactWs w;
  const int B = kv->B;
  w.ctrl = c.take<CompactCtrl>(1);
  w.pb = c.take<int32_t>(B);
  w.n_new = c.take<int32_t>(B);
  w.old_blocks = c.take<int32_t>(B);
  w.new_ctx = c.take<int32_t>(B);
  w.old_ctx = c.take<int32_t>(B);
  w.off_new = c.take<int32_t>(B);
  w.push_count = c.take<int32_t>(B);
  w.newpage = c.take<int32_t>((size_t)B * kv->max_pages_per_seq);
  w.row = (int64_t)max_keep + kv->page_size;
  w.slot_tmp = c.take<int32_t>((size_t)B * kv->Hkv * w.row);
  w.aux_tmp = aux ? c.take<float>((size_t)B * kv->Hkv * w.row) : nullptr;
  if (!aux) c.take<float>((size_t)B * kv->Hkv * w.row);  // size does not depend on aux
  *bytes = c.bytes();
  return w;
}

// Records sequence b's fresh pages for the commit and counts its old pages
// from the first rewritten block on that go back to the free list (a busy
// page only loses a reference), into push_count[b] (zeroed by the plan).
// Share `part` of `parts`: every thread of `parts` CTAs calls it, each CTA
// with its own part.
SE_DEV void record_fresh_pages(const se_paged_kv& kv, const CompactWs& w, int b, int part = 0,
                               int parts = 1) {
  __shared__ int s_cnt;
  if (threadIdx.x == 0) s_cnt = 0;
  __syncthreads();
  const int step = parts * blockDim.x;
  const int first = part * blockDim.x + threadIdx.x;
  const int pop0 = w.ctrl->top0 - 1 - w.off_new[b];
  for (int i = first; i < w.n_new[b]; i += step) w.newpage[w.off_new[b] + i] = kv.free_list[pop0 - i];
  const int32_t* btb = kv.block_table + (int64_t)b * kv.max_pages_per_seq;
  int cnt = 0;
  for (int blk = w.pb[b] + first; blk < w.old_blocks[b]; blk += step) {
    const int page = btb[blk];
    cnt += (page >= 0 && (kv.page_refcount == nullptr || kv.page_refcount[page] <= 1)) ? 1 : 0;
  }
  if (cnt) atomicAdd(&s_cnt, cnt);
  __syncthreads();
  if (threadIdx.x == 0 && s_cnt) atomicAdd(&w.push_count[b], s_cnt);
}

}  // namespace se
