// Host block manager: which physical blocks hold each sequence's keys and values.
// The operations and the policies they follow are stated in pa_block_manager.h.
//
// Data structures, all O(1) per block touched:
//  - the idle-block queue is an intrusive doubly linked list over block ids (a block is
//    in it exactly when no sequence reads it), so a prefix-cache hit can take a block
//    out of the middle;
//  - keys of cached blocks map to block ids in a hash table (sha256 digests are uniform,
//    so their first 8 bytes serve as the table's hash);
//  - a sequence keeps its block ids, the keys of its full blocks (with prefix caching)
//    and the token ids of its partly filled last block (the only ones a later key needs).
#include <algorithm>
#include <array>
#include <deque>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include <string.h>

#include "pa_block_manager.h"
#include "pa_internal.h"
#include "pa_sha256.h"

namespace {

using Key = std::array<uint8_t, 32>;

struct KeyHash {
  size_t operator()(const Key& k) const {
    uint64_t h;
    memcpy(&h, k.data(), sizeof(h));
    return (size_t)h;
  }
};

struct Seq {
  std::vector<int32_t> blocks;  // device ids, or host ids while swapped out
  std::vector<Key> keys;        // keys of the full blocks (prefix caching only)
  std::vector<int32_t> tail;    // token ids of the partly filled last block
  int64_t tokens = 0;
  std::string extra;
  bool swapped = false;
  uint64_t batch = 0;  // last batched call that listed the sequence
};

}  // namespace

struct pa_block_manager {
  int nb, bs;
  bool caching;
  // idle queue: ids 0..nb-1, sentinel nb
  std::vector<int32_t> next, prev;
  int queued = 0;
  std::vector<int32_t> ref;
  std::vector<uint8_t> has_key;
  std::vector<Key> key;
  std::unordered_map<Key, int32_t, KeyHash> cached;
  std::deque<int32_t> host_free;
  std::vector<int32_t> host_ref;
  std::unordered_map<int64_t, Seq> seqs;
  std::vector<int32_t> copies;  // (src, dst) flattened
  uint64_t batches = 0;         // batched calls so far
  std::vector<Seq*> batch_seqs;
  std::vector<std::pair<int32_t, int32_t>> batch_copied;  // source block, copies counted

  pa_block_manager(int num_blocks, int block_size, bool prefix_caching, int num_host)
      : nb(num_blocks), bs(block_size), caching(prefix_caching), next(num_blocks + 1),
        prev(num_blocks + 1), ref(num_blocks, 0), has_key(num_blocks, 0), key(num_blocks),
        host_ref(num_host, 0) {
    next[nb] = prev[nb] = nb;
    for (int b = 0; b < nb; ++b) push_back(b);
    for (int h = 0; h < num_host; ++h) host_free.push_back(h);
  }

  // ------------------------------------------------------------------ idle queue
  void push_back(int32_t b) {
    const int32_t last = prev[nb];
    next[last] = b;
    prev[b] = last;
    next[b] = nb;
    prev[nb] = b;
    ++queued;
  }
  void unlink(int32_t b) {
    next[prev[b]] = next[b];
    prev[next[b]] = prev[b];
    --queued;
  }
  // Takes the least recently used idle block (evicting its key) with one reader.
  int32_t take() {
    const int32_t b = next[nb];
    unlink(b);
    if (has_key[b]) {
      cached.erase(key[b]);
      has_key[b] = 0;
    }
    ref[b] = 1;
    return b;
  }
  void release(int32_t b) {
    if (--ref[b] == 0) push_back(b);
  }

  // ------------------------------------------------------------------ keys
  Key block_key(const Key* parent, const int32_t* toks, const std::string& extra) const {
    std::vector<uint8_t> msg(32 + 4 * (size_t)bs + extra.size(), 0);
    if (parent) memcpy(msg.data(), parent->data(), 32);
    for (int i = 0; i < bs; ++i) {  // little-endian int32
      const uint32_t v = (uint32_t)toks[i];
      msg[32 + 4 * i] = (uint8_t)v;
      msg[32 + 4 * i + 1] = (uint8_t)(v >> 8);
      msg[32 + 4 * i + 2] = (uint8_t)(v >> 16);
      msg[32 + 4 * i + 3] = (uint8_t)(v >> 24);
    }
    if (!extra.empty()) memcpy(msg.data() + 32 + 4 * (size_t)bs, extra.data(), extra.size());
    Key k;
    pa::sha256(msg.data(), msg.size(), k.data());
    return k;
  }
  // Block i of s became full with key k: register it unless the key is held already.
  void on_full(Seq& s, size_t i, const Key& k) {
    s.keys.push_back(k);
    const int32_t b = s.blocks[i];
    if (!has_key[b] && cached.find(k) == cached.end()) {
      cached.emplace(k, b);
      key[b] = k;
      has_key[b] = 1;
    }
  }

  // Appends n tokens to s; the caller has checked that the pool can supply the blocks.
  void append(Seq& s, const int32_t* toks, int n) {
    for (int i = 0; i < n; ++i) {
      const int64_t pos = s.tokens;
      if (pos % bs == 0) {
        s.blocks.push_back(take());
      } else if (ref[s.blocks.back()] > 1) {  // copy-on-write
        const int32_t src = s.blocks.back();
        const int32_t dst = take();
        copies.push_back(src);
        copies.push_back(dst);
        --ref[src];
        s.blocks.back() = dst;
      }
      s.tail.push_back(toks[i]);
      ++s.tokens;
      if ((pos + 1) % bs == 0) {
        if (caching) {
          const size_t bi = (size_t)(pos / bs);
          const Key k = block_key(bi ? &s.keys[bi - 1] : nullptr, s.tail.data(), s.extra);
          on_full(s, bi, k);
        }
        s.tail.clear();
      }
    }
  }

  Seq* resident(int64_t id, const char* fn) {
    auto it = seqs.find(id);
    if (it == seqs.end()) {
      pa::fail(PA_ERR_INVALID_ARG, "%s: unknown sequence %lld", fn, (long long)id);
      return nullptr;
    }
    if (it->second.swapped) {
      pa::fail(PA_ERR_INVALID_ARG, "%s: sequence %lld is swapped out", fn, (long long)id);
      return nullptr;
    }
    return &it->second;
  }
};

namespace {
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
}  // namespace

extern "C" {

int pa_bm_create(int num_blocks, int block_size, int prefix_caching, int num_host_blocks,
                 pa_block_manager** out) {
  pa::clear_error();
  if (!out) return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_create: null output pointer");
  *out = nullptr;
  if (num_blocks <= 0 || block_size <= 0 || num_host_blocks < 0)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_create: num_blocks and block_size must be > 0");
  try {
    *out = new pa_block_manager(num_blocks, block_size, prefix_caching != 0, num_host_blocks);
  } catch (...) {
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_create: out of host memory");
  }
  return PA_OK;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int pa_bm_num_free_blocks(const pa_block_manager* bm) { return bm ? bm->queued : -1; }

int pa_bm_num_free_host_blocks(const pa_block_manager* bm) {
  return bm ? (int)bm->host_free.size() : -1;
}

int pa_bm_can_allocate(const pa_block_manager* bm, int num_tokens, int watermark_blocks) {
  if (!bm || num_tokens < 0) return 0;
  return cdiv(num_tokens, bm->bs) + watermark_blocks <= bm->queued ? 1 : 0;
}

int pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens,
                       int num_tokens, const void* extra, int extra_bytes, int* cached_tokens) {
  pa::clear_error();
  if (!bm || !tokens || num_tokens <= 0 || extra_bytes < 0 || (extra_bytes > 0 && !extra))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_add_sequence: bad arguments");
  if (bm->seqs.count(seq_id))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_add_sequence: sequence %lld exists",
                    (long long)seq_id);
  const int bs = bm->bs;
  const int64_t nfull = num_tokens / bs, nblocks = cdiv(num_tokens, bs);
  std::string ex(static_cast<const char*>(extra), static_cast<const char*>(extra) + extra_bytes);
  std::vector<Key> chain;
  std::vector<int32_t> hits;
  if (bm->caching) {
    chain.reserve(nfull);
    bool hitting = true;
    for (int64_t i = 0; i < nfull; ++i) {
      chain.push_back(bm->block_key(i ? &chain[i - 1] : nullptr, tokens + i * bs, ex));
      if (hitting) {
        auto it = bm->cached.find(chain.back());
        if (it == bm->cached.end()) hitting = false;
        else hits.push_back(it->second);
      }
    }
  }
  int64_t idle_hits = 0;
  for (int32_t b : hits) idle_hits += bm->ref[b] == 0;
  if (nblocks - (int64_t)hits.size() > bm->queued - idle_hits)
    return pa::fail(PA_ERR_NO_BLOCKS, "pa_bm_add_sequence: %lld blocks needed, %d free",
                    (long long)(nblocks - (int64_t)hits.size()), bm->queued - (int)idle_hits);
  Seq s;
  s.extra = std::move(ex);
  s.tokens = num_tokens;
  s.blocks.reserve(nblocks);
  for (int32_t b : hits) {
    if (bm->ref[b] == 0) bm->unlink(b);
    ++bm->ref[b];
    s.blocks.push_back(b);
  }
  while ((int64_t)s.blocks.size() < nblocks) s.blocks.push_back(bm->take());
  if (bm->caching)
    for (int64_t i = 0; i < nfull; ++i) bm->on_full(s, (size_t)i, chain[i]);
  s.tail.assign(tokens + nfull * bs, tokens + num_tokens);
  bm->seqs.emplace(seq_id, std::move(s));
  if (cached_tokens) *cached_tokens = (int)hits.size() * bs;
  return PA_OK;
}

int pa_bm_append_tokens(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens, int n) {
  pa::clear_error();
  if (!bm || n < 0 || (n > 0 && !tokens))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_append_tokens: bad arguments");
  Seq* s = bm->resident(seq_id, "pa_bm_append_tokens");
  if (!s) return PA_ERR_INVALID_ARG;
  if (n == 0) return PA_OK;
  const int bs = bm->bs;
  const int64_t n0 = s->tokens;
  int64_t need = cdiv(n0 + n, bs) - cdiv(n0, bs);
  if (n0 % bs != 0 && bm->ref[s->blocks.back()] > 1) ++need;
  if (need > bm->queued)
    return pa::fail(PA_ERR_NO_BLOCKS, "pa_bm_append_tokens: %lld blocks needed, %d free",
                    (long long)need, bm->queued);
  bm->append(*s, tokens, n);
  return PA_OK;
}

int pa_bm_append_tokens_batch(pa_block_manager* bm, const int64_t* seq_ids, int n,
                              const int32_t* tokens, const int32_t* counts) {
  pa::clear_error();
  if (!bm || n < 0 || (n > 0 && !seq_ids))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_append_tokens_batch: bad arguments");
  // dry run: every sequence resident and listed once, and the blocks the whole batch
  // takes, copies included (a copy lowers its source's reference count, so later
  // sequences in the batch may append in place)
  const uint64_t stamp = ++bm->batches;
  bm->batch_seqs.resize(n);
  bm->batch_copied.clear();
  int64_t need = 0, total = 0;
  for (int i = 0; i < n; ++i) {
    Seq* s = bm->resident(seq_ids[i], "pa_bm_append_tokens_batch");
    if (!s) return PA_ERR_INVALID_ARG;
    if (s->batch == stamp)
      return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_append_tokens_batch: sequence %lld repeated",
                      (long long)seq_ids[i]);
    s->batch = stamp;
    const int k = counts ? counts[i] : 1;
    if (k < 0) return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_append_tokens_batch: negative count");
    bm->batch_seqs[i] = s;
    total += k;
    if (k == 0) continue;
    const int64_t n0 = s->tokens;
    need += cdiv(n0 + k, bm->bs) - cdiv(n0, bm->bs);
    if (n0 % bm->bs != 0 && bm->ref[s->blocks.back()] > 1) {  // shared partly filled block
      const int32_t last = s->blocks.back();
      int32_t c = 0;
      for (auto& bc : bm->batch_copied)
        if (bc.first == last) c = bc.second;
      if (bm->ref[last] - c > 1) {
        ++need;
        bool found = false;
        for (auto& bc : bm->batch_copied)
          if (bc.first == last) { ++bc.second; found = true; }
        if (!found) bm->batch_copied.emplace_back(last, 1);
      }
    }
  }
  if (total > 0 && !tokens)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_append_tokens_batch: null tokens");
  if (need > bm->queued)
    return pa::fail(PA_ERR_NO_BLOCKS, "pa_bm_append_tokens_batch: %lld blocks needed, %d free",
                    (long long)need, bm->queued);
  const int32_t* t = tokens;
  for (int i = 0; i < n; ++i) {
    const int k = counts ? counts[i] : 1;
    bm->append(*bm->batch_seqs[i], t, k);
    t += k;
  }
  return PA_OK;
}

int pa_bm_fork(pa_block_manager* bm, int64_t parent_id, int64_t child_id) {
  pa::clear_error();
  if (!bm) return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_fork: null manager");
  Seq* p = bm->resident(parent_id, "pa_bm_fork");
  if (!p) return PA_ERR_INVALID_ARG;
  if (bm->seqs.count(child_id))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_fork: sequence %lld exists", (long long)child_id);
  Seq c = *p;  // copy before inserting (the insertion may move *p)
  for (int32_t b : c.blocks) ++bm->ref[b];
  bm->seqs.emplace(child_id, std::move(c));
  return PA_OK;
}

int pa_bm_free_sequence(pa_block_manager* bm, int64_t seq_id) {
  pa::clear_error();
  if (!bm) return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_free_sequence: null manager");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end())
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_free_sequence: unknown sequence %lld",
                    (long long)seq_id);
  const Seq& s = it->second;
  for (auto b = s.blocks.rbegin(); b != s.blocks.rend(); ++b) {  // tail first
    if (s.swapped) {
      if (--bm->host_ref[*b] == 0) bm->host_free.push_back(*b);
    } else {
      bm->release(*b);
    }
  }
  bm->seqs.erase(it);
  return PA_OK;
}

int pa_bm_take_copies(pa_block_manager* bm, int32_t* pairs, int max_pairs, int* num_pairs) {
  pa::clear_error();
  if (!bm || !num_pairs || max_pairs < 0)
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_take_copies: bad arguments");
  const int n = (int)(bm->copies.size() / 2);
  *num_pairs = n;
  if (n > max_pairs || (n > 0 && !pairs))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_take_copies: %d pairs, room for %d", n,
                    max_pairs);
  if (n) memcpy(pairs, bm->copies.data(), sizeof(int32_t) * 2 * n);
  bm->copies.clear();
  return PA_OK;
}

namespace {
// The listed sequences, checked to exist, be distinct and be in the wanted state; and
// their distinct blocks in order of first appearance.
int gather(pa_block_manager* bm, const int64_t* ids, int n, bool swapped, const char* fn,
           std::vector<Seq*>& seqs, std::vector<int32_t>& blocks) {
  if (!ids || n < 0) return pa::fail(PA_ERR_INVALID_ARG, "%s: bad arguments", fn);
  std::unordered_set<int64_t> seen_ids;
  std::unordered_set<int32_t> seen;
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(ids[i]);
    if (it == bm->seqs.end() || !seen_ids.insert(ids[i]).second)
      return pa::fail(PA_ERR_INVALID_ARG, "%s: unknown or repeated sequence %lld", fn,
                      (long long)ids[i]);
    if (it->second.swapped != swapped)
      return pa::fail(PA_ERR_INVALID_ARG, "%s: sequence %lld is %s", fn, (long long)ids[i],
                      swapped ? "resident" : "swapped out");
    seqs.push_back(&it->second);
    for (int32_t b : it->second.blocks)
      if (seen.insert(b).second) blocks.push_back(b);
  }
  return PA_OK;
}
}  // namespace

int pa_bm_swap_out(pa_block_manager* bm, const int64_t* seq_ids, int n, int32_t* pairs,
                   int max_pairs, int* num_pairs) {
  pa::clear_error();
  if (!bm || !num_pairs) return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_swap_out: bad arguments");
  std::vector<Seq*> seqs;
  std::vector<int32_t> blocks;
  int rc = gather(bm, seq_ids, n, false, "pa_bm_swap_out", seqs, blocks);
  if (rc != PA_OK) return rc;
  *num_pairs = (int)blocks.size();
  if ((int)blocks.size() > max_pairs || (!blocks.empty() && !pairs))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_swap_out: %zu pairs, room for %d", blocks.size(),
                    max_pairs);
  if (blocks.size() > bm->host_free.size())
    return pa::fail(PA_ERR_NO_BLOCKS, "pa_bm_swap_out: %zu host blocks needed, %zu free",
                    blocks.size(), bm->host_free.size());
  std::unordered_map<int32_t, int32_t> to_host;
  for (size_t i = 0; i < blocks.size(); ++i) {
    const int32_t h = bm->host_free.front();
    bm->host_free.pop_front();
    to_host[blocks[i]] = h;
    pairs[2 * i] = blocks[i];
    pairs[2 * i + 1] = h;
  }
  for (Seq* s : seqs) {
    for (auto b = s->blocks.rbegin(); b != s->blocks.rend(); ++b) {
      ++bm->host_ref[to_host[*b]];
      bm->release(*b);
    }
    for (int32_t& b : s->blocks) b = to_host[b];
    s->swapped = true;
  }
  return PA_OK;
}

int pa_bm_swap_in(pa_block_manager* bm, const int64_t* seq_ids, int n, int32_t* pairs,
                  int max_pairs, int* num_pairs) {
  pa::clear_error();
  if (!bm || !num_pairs) return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_swap_in: bad arguments");
  std::vector<Seq*> seqs;
  std::vector<int32_t> blocks;
  int rc = gather(bm, seq_ids, n, true, "pa_bm_swap_in", seqs, blocks);
  if (rc != PA_OK) return rc;
  *num_pairs = (int)blocks.size();
  if ((int)blocks.size() > max_pairs || (!blocks.empty() && !pairs))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_swap_in: %zu pairs, room for %d", blocks.size(),
                    max_pairs);
  if ((int)blocks.size() > bm->queued)
    return pa::fail(PA_ERR_NO_BLOCKS, "pa_bm_swap_in: %zu blocks needed, %d free", blocks.size(),
                    bm->queued);
  std::unordered_map<int32_t, int32_t> to_dev;
  for (size_t i = 0; i < blocks.size(); ++i) {
    const int32_t d = bm->take();
    bm->ref[d] = 0;
    to_dev[blocks[i]] = d;
    pairs[2 * i] = blocks[i];
    pairs[2 * i + 1] = d;
  }
  for (Seq* s : seqs) {
    for (auto h = s->blocks.rbegin(); h != s->blocks.rend(); ++h) {
      ++bm->ref[to_dev[*h]];
      if (--bm->host_ref[*h] == 0) bm->host_free.push_back(*h);
    }
    for (int32_t& h : s->blocks) h = to_dev[h];
    s->swapped = false;
  }
  return PA_OK;
}

int pa_bm_num_tokens(const pa_block_manager* bm, int64_t seq_id) {
  if (!bm) return -1;
  auto it = bm->seqs.find(seq_id);
  return it == bm->seqs.end() ? -1 : (int)it->second.tokens;
}

int pa_bm_block_tables(const pa_block_manager* bm, const int64_t* seq_ids, int n, int width,
                       int32_t* tables, int32_t* context_lens) {
  pa::clear_error();
  if (!bm || n < 0 || width < 0 || (n > 0 && (!seq_ids || !tables || !context_lens)))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_block_tables: bad arguments");
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end() || it->second.swapped)
      return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_block_tables: sequence %lld not resident",
                      (long long)seq_ids[i]);
    if ((int64_t)it->second.blocks.size() > width)
      return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_block_tables: %zu blocks wider than %d",
                      it->second.blocks.size(), width);
  }
  for (int i = 0; i < n; ++i) {
    const Seq& s = bm->seqs.find(seq_ids[i])->second;
    int32_t* row = tables + (size_t)i * width;
    std::copy(s.blocks.begin(), s.blocks.end(), row);
    std::fill(row + s.blocks.size(), row + width, -1);
    context_lens[i] = (int32_t)s.tokens;
  }
  return PA_OK;
}

int pa_bm_slot_mapping(const pa_block_manager* bm, const int64_t* seq_ids, int n,
                       const int32_t* query_lens, int64_t* slots, int max_slots,
                       int* num_slots) {
  pa::clear_error();
  if (!bm || n < 0 || !num_slots || (n > 0 && (!seq_ids || !query_lens)))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_slot_mapping: bad arguments");
  int64_t total = 0;
  for (int i = 0; i < n; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end() || it->second.swapped)
      return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_slot_mapping: sequence %lld not resident",
                      (long long)seq_ids[i]);
    if (query_lens[i] < 0 || query_lens[i] > it->second.tokens)
      return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_slot_mapping: query length %d of %lld tokens",
                      query_lens[i], (long long)it->second.tokens);
    total += query_lens[i];
  }
  *num_slots = (int)total;
  if (total > max_slots || (total > 0 && !slots))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_slot_mapping: %lld slots, room for %d",
                    (long long)total, max_slots);
  int64_t o = 0;
  for (int i = 0; i < n; ++i) {
    const Seq& s = bm->seqs.find(seq_ids[i])->second;
    for (int64_t pos = s.tokens - query_lens[i]; pos < s.tokens; ++pos)
      slots[o++] = (int64_t)s.blocks[pos / bm->bs] * bm->bs + pos % bm->bs;
  }
  return PA_OK;
}

int pa_bm_refcount(const pa_block_manager* bm, int block) {
  return (bm && block >= 0 && block < bm->nb) ? bm->ref[block] : -1;
}

int pa_bm_is_cached(const pa_block_manager* bm, int block) {
  return (bm && block >= 0 && block < bm->nb) ? (int)bm->has_key[block] : -1;
}

int pa_bm_free_queue(const pa_block_manager* bm, int32_t* out, int max, int* n) {
  pa::clear_error();
  if (!bm || !n) return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_free_queue: bad arguments");
  *n = bm->queued;
  if (bm->queued > max || (bm->queued > 0 && !out))
    return pa::fail(PA_ERR_INVALID_ARG, "pa_bm_free_queue: %d blocks, room for %d", bm->queued,
                    max);
  int i = 0;
  for (int32_t b = bm->next[bm->nb]; b != bm->nb; b = bm->next[b]) out[i++] = b;
  return PA_OK;
}

void pa_sha256(const void* data, size_t n, uint8_t digest[32]) { pa::sha256(data, n, digest); }

}  // extern "C"
