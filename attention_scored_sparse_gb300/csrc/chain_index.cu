// Chain index: which sequence row of the paged cache holds which session.
//
// SparseEngine "How it differs" (Chain Cache): eviction-based methods break
// the assumption that every token of a prefix is resident, but eviction
// never changes a sequence's logical prefix.  The index ties each session
// (chain_id) to the cache row that holds its retained KV and to its logical
// token prefix; a request whose tokens start with an idle chain's prefix
// resumes that chain's row and prefills only the rest; idle chains are
// reclaimed least-recently-used first when a row is needed.
//
// Host code only (no device work): the caller releases a reclaimed row's
// pages with se_release_seqs.  Readings where the pages are silent: the
// longest matching prefix wins (ties: most recently used); a new chain takes
// the lowest free row, else the least recently used idle chain's row; acquire
// and finish both count as use; chain ids count up from 1.  All calls on one
// index are serialised by a mutex.
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "se.h"

struct se_chain_index {
  struct Chain {
    int32_t row;
    std::vector<int32_t> tokens;   // logical prefix
    bool busy;
    uint64_t used;
  };
  std::mutex mu;
  std::vector<int64_t> rows;       // row -> chain id, 0 = free
  std::unordered_map<int64_t, Chain> chains;
  int64_t next_id = 1;
  uint64_t clock = 0;
};

extern "C" se_chain_index* se_chain_index_create(int32_t n_rows) {
  if (n_rows < 1) return nullptr;
  se_chain_index* idx = new (std::nothrow) se_chain_index();
  if (idx == nullptr) return nullptr;
  idx->rows.assign((size_t)n_rows, 0);
  return idx;
}

extern "C" void se_chain_index_destroy(se_chain_index* idx) { delete idx; }

extern "C" se_status se_chain_acquire(se_chain_index* idx, const int32_t* tokens, int64_t n_tokens,
                                      int64_t* chain_id, int32_t* row, int64_t* reuse_len,
                                      int32_t* reclaimed_row) {
  if (idx == nullptr || chain_id == nullptr || row == nullptr || reuse_len == nullptr ||
      reclaimed_row == nullptr || n_tokens < 0 || (n_tokens > 0 && tokens == nullptr))
    return SE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(idx->mu);
  // resume: the idle chain with the longest prefix of the request
  int64_t best = 0;
  size_t best_len = 0;
  uint64_t best_used = 0;
  for (auto& kv : idx->chains) {
    const auto& ch = kv.second;
    if (ch.busy || ch.tokens.size() > (size_t)n_tokens) continue;
    if (!ch.tokens.empty() &&
        std::memcmp(ch.tokens.data(), tokens, ch.tokens.size() * sizeof(int32_t)) != 0)
      continue;
    const size_t len = ch.tokens.size();
    if (best == 0 || len > best_len || (len == best_len && ch.used > best_used)) {
      best = kv.first;
      best_len = len;
      best_used = ch.used;
    }
  }
  if (best != 0) {
    auto& ch = idx->chains[best];
    ch.busy = true;
    ch.used = ++idx->clock;
    *chain_id = best;
    *row = ch.row;
    *reuse_len = (int64_t)ch.tokens.size();
    *reclaimed_row = -1;
    return SE_OK;
  }
  // a new chain: lowest free row, else the least recently used idle chain's
  int32_t r = -1, reclaimed = -1;
  for (size_t i = 0; i < idx->rows.size(); ++i)
    if (idx->rows[i] == 0) {
      r = (int32_t)i;
      break;
    }
  if (r < 0) {
    int64_t victim = 0;
    uint64_t oldest = 0;
    for (auto& kv : idx->chains)
      if (!kv.second.busy && (victim == 0 || kv.second.used < oldest)) {
        victim = kv.first;
        oldest = kv.second.used;
      }
    if (victim == 0) return SE_ERR_BUSY;   // every row is serving a request
    r = idx->chains[victim].row;
    idx->chains.erase(victim);
    reclaimed = r;
  }
  const int64_t id = idx->next_id++;
  idx->chains[id] = se_chain_index::Chain{r, {}, true, ++idx->clock};
  idx->rows[(size_t)r] = id;
  *chain_id = id;
  *row = r;
  *reuse_len = 0;
  *reclaimed_row = reclaimed;
  return SE_OK;
}

extern "C" se_status se_chain_finish(se_chain_index* idx, int64_t chain_id, const int32_t* tokens,
                                     int64_t n_tokens) {
  if (idx == nullptr || n_tokens < 0 || (n_tokens > 0 && tokens == nullptr))
    return SE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(idx->mu);
  auto it = idx->chains.find(chain_id);
  if (it == idx->chains.end() || !it->second.busy) return SE_ERR_INVALID_ARG;
  it->second.tokens.assign(tokens, tokens + n_tokens);
  it->second.busy = false;
  it->second.used = ++idx->clock;
  return SE_OK;
}

extern "C" se_status se_chain_drop(se_chain_index* idx, int64_t chain_id, int32_t* row) {
  if (idx == nullptr || row == nullptr) return SE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(idx->mu);
  auto it = idx->chains.find(chain_id);
  if (it == idx->chains.end() || it->second.busy) return SE_ERR_INVALID_ARG;
  *row = it->second.row;
  idx->rows[(size_t)it->second.row] = 0;
  idx->chains.erase(it);
  return SE_OK;
}

extern "C" int32_t se_chain_count(se_chain_index* idx) {
  if (idx == nullptr) return 0;
  std::lock_guard<std::mutex> lock(idx->mu);
  return (int32_t)idx->chains.size();
}
