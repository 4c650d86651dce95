// Host side of span reuse: the block-hash chain with span separators and the
// prefix cache that turns a request's block hashes into its block table and
// block starts (MiniPIC summary, gist.science 2606.13126, section 2.2).
//
// Hash of full block i of a prompt (tokens x_i, block_size of them):
//   default  h_i = H(h_{i-1}, x_i), h_{-1} = h_0
//   SSEP     h_i = H(h_0, x_i)        when x_i starts with the SSEP token
//   PDEP     h_i = H(h_0, x_{<=i})    when x_i starts with the PDEP token
// with H(p, t) the 64-bit FNV-1a hash of p (8 bytes, little endian) followed by
// the tokens t (4 bytes each, little endian).  FNV-1a is a streaming hash, so
// H(h_0, x_{<=i}) is kept as one running state over the prompt.
//
// The prefix cache maps a full block's hash to a physical block.  A request's
// block b gets logical start b * block_size: because keys are stored unrotated,
// a physical block found in the cache is read at this request's offset,
// whatever offset the request that computed it had.  Misses take a
// never-used block, else evict the unreferenced cached block released longest
// ago; a request that does not fit leaves the cache as it was.  Host code only.
#include <cstdint>
#include <map>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/minipic.h"

namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001b3ull;

inline uint64_t fnv_byte(uint64_t h, uint32_t b) { return (h ^ (b & 0xffu)) * kFnvPrime; }

inline uint64_t fnv_u64(uint64_t h, uint64_t v) {
  for (int i = 0; i < 8; ++i) h = fnv_byte(h, (uint32_t)(v >> (8 * i)));
  return h;
}

inline uint64_t fnv_i32(uint64_t h, int32_t t) {
  const uint32_t u = (uint32_t)t;
  for (int i = 0; i < 4; ++i) h = fnv_byte(h, u >> (8 * i));
  return h;
}

inline uint64_t chain_hash(uint64_t parent, const int32_t* x, int32_t n) {
  uint64_t h = fnv_u64(kFnvOffset, parent);
  for (int32_t k = 0; k < n; ++k) h = fnv_i32(h, x[k]);
  return h;
}

}  // namespace

struct minipic_prefix_cache {
  int32_t num_blocks = 0;
  int32_t next_fresh = 0;
  uint64_t stamp = 0;                               // release counter
  std::unordered_map<uint64_t, int32_t> by_hash;    // hash -> block
  std::vector<uint64_t> hash_of;                    // block -> hash (when cached)
  std::vector<uint8_t> cached;                      // block has a hash entry
  std::vector<int32_t> refs;
  std::vector<uint64_t> stamp_of;                   // block -> its release stamp (when released)
  std::map<uint64_t, int32_t> released;             // stamp -> unreferenced block, oldest first
};

namespace {

// One change made while assigning a request, undone in reverse order when the
// request does not fit.
struct Undo {
  enum Kind { kFresh, kEvict, kUnrelease, kInsertHash, kRef } kind;
  int32_t block;
  uint64_t stamp;
  uint64_t hash;
  bool had_hash;
};

// A block for a miss, or -1: never-used first, else the oldest released one
// (its hash entry is dropped).
int32_t take_block(minipic_prefix_cache* c, std::vector<Undo>& log) {
  if (c->next_fresh < c->num_blocks) {
    log.push_back({Undo::kFresh, c->next_fresh, 0, 0, false});
    return c->next_fresh++;
  }
  if (c->released.empty()) return -1;
  const auto it = c->released.begin();
  const int32_t b = it->second;
  Undo u{Undo::kEvict, b, it->first, c->hash_of[b], c->cached[b] != 0};
  c->released.erase(it);
  if (u.had_hash) {
    c->by_hash.erase(u.hash);
    c->cached[b] = 0;
  }
  log.push_back(u);
  return b;
}

void rollback(minipic_prefix_cache* c, std::vector<Undo>& log) {
  for (auto it = log.rbegin(); it != log.rend(); ++it) {
    const Undo& u = *it;
    switch (u.kind) {
      case Undo::kFresh: --c->next_fresh; break;
      case Undo::kEvict:
        c->released.emplace(u.stamp, u.block);
        c->stamp_of[u.block] = u.stamp;
        if (u.had_hash) {
          c->by_hash[u.hash] = u.block;
          c->hash_of[u.block] = u.hash;
          c->cached[u.block] = 1;
        }
        break;
      case Undo::kUnrelease:
        c->released.emplace(u.stamp, u.block);
        c->stamp_of[u.block] = u.stamp;
        break;
      case Undo::kInsertHash:
        c->by_hash.erase(u.hash);
        c->cached[u.block] = 0;
        break;
      case Undo::kRef: --c->refs[u.block]; break;
    }
  }
  log.clear();
}

}  // namespace

extern "C" {

minipic_status minipic_block_hashes(const int32_t* tokens, int32_t n_tokens, int32_t block_size, int32_t ssep_token,
                                    int32_t pdep_token, uint64_t h0, uint64_t* hashes, int32_t max_hashes,
                                    int32_t* n_hashes) {
  if (n_tokens < 0 || block_size <= 0 || max_hashes < 0 || !n_hashes) return MINIPIC_ERR_INVALID;
  if (n_tokens > 0 && !tokens) return MINIPIC_ERR_INVALID;
  const int32_t n_full = n_tokens / block_size;
  if (n_full > max_hashes || (n_full > 0 && !hashes)) return MINIPIC_ERR_INVALID;
  uint64_t prev = h0;
  uint64_t run = fnv_u64(kFnvOffset, h0);  // H(h_0, tokens so far), extended block by block
  for (int32_t i = 0; i < n_full; ++i) {
    const int32_t* x = tokens + (size_t)i * block_size;
    for (int32_t k = 0; k < block_size; ++k) run = fnv_i32(run, x[k]);
    uint64_t h;
    if (x[0] == ssep_token) h = chain_hash(h0, x, block_size);
    else if (x[0] == pdep_token) h = run;
    else h = chain_hash(prev, x, block_size);
    hashes[i] = h;
    prev = h;
  }
  *n_hashes = n_full;
  return MINIPIC_OK;
}

minipic_status minipic_prefix_cache_create(int32_t num_blocks, minipic_prefix_cache** cache) {
  if (num_blocks <= 0 || !cache) return MINIPIC_ERR_INVALID;
  minipic_prefix_cache* c = new (std::nothrow) minipic_prefix_cache();
  if (!c) return MINIPIC_ERR_CAPACITY;
  try {
    c->num_blocks = num_blocks;
    c->hash_of.assign(num_blocks, 0);
    c->cached.assign(num_blocks, 0);
    c->refs.assign(num_blocks, 0);
    c->stamp_of.assign(num_blocks, 0);
  } catch (...) {
    delete c;
    return MINIPIC_ERR_CAPACITY;
  }
  *cache = c;
  return MINIPIC_OK;
}

void minipic_prefix_cache_destroy(minipic_prefix_cache* cache) { delete cache; }

minipic_status minipic_prefix_cache_assign(minipic_prefix_cache* c, const uint64_t* hashes, int32_t n_hashed,
                                           int32_t n_blocks, int32_t block_size, int32_t* block_table,
                                           int32_t* block_starts, uint8_t* is_new) {
  if (!c || n_hashed < 0 || n_blocks < 0 || n_hashed > n_blocks || block_size <= 0) return MINIPIC_ERR_INVALID;
  if ((n_hashed > 0 && !hashes) || (n_blocks > 0 && (!block_table || !block_starts || !is_new)))
    return MINIPIC_ERR_INVALID;
  if ((int64_t)n_blocks * block_size > INT32_MAX) return MINIPIC_ERR_INVALID;
  std::vector<Undo> log;
  try {
    for (int32_t b = 0; b < n_blocks; ++b) {
      int32_t blk = -1;
      bool fresh = true;
      if (b < n_hashed) {
        const auto f = c->by_hash.find(hashes[b]);
        if (f != c->by_hash.end()) {
          blk = f->second;
          fresh = false;
          if (c->refs[blk] == 0) {  // a released cached block: back in use
            const uint64_t st = c->stamp_of[blk];
            c->released.erase(st);
            log.push_back({Undo::kUnrelease, blk, st, 0, false});
          }
        }
      }
      if (fresh) {
        blk = take_block(c, log);
        if (blk < 0) {
          rollback(c, log);
          return MINIPIC_ERR_CAPACITY;
        }
        if (b < n_hashed) {
          c->by_hash[hashes[b]] = blk;
          c->hash_of[blk] = hashes[b];
          c->cached[blk] = 1;
          log.push_back({Undo::kInsertHash, blk, 0, hashes[b], false});
        }
      }
      ++c->refs[blk];
      log.push_back({Undo::kRef, blk, 0, 0, false});
      block_table[b] = blk;
      block_starts[b] = b * block_size;
      is_new[b] = fresh ? 1 : 0;
    }
  } catch (...) {
    rollback(c, log);
    return MINIPIC_ERR_CAPACITY;
  }
  return MINIPIC_OK;
}

minipic_status minipic_prefix_cache_release(minipic_prefix_cache* c, const int32_t* block_ids, int32_t n) {
  if (!c || n < 0 || (n > 0 && !block_ids)) return MINIPIC_ERR_INVALID;
  for (int32_t i = 0; i < n; ++i) {  // validate first: nothing changes on a bad id
    const int32_t b = block_ids[i];
    if (b < 0 || b >= c->num_blocks || c->refs[b] <= 0) return MINIPIC_ERR_INVALID;
  }
  std::vector<int32_t> dec(n > 0 ? n : 0);
  for (int32_t i = 0; i < n; ++i) dec[i] = block_ids[i];
  // a block listed k times needs at least k references
  std::unordered_map<int32_t, int32_t> count;
  for (int32_t b : dec) ++count[b];
  for (const auto& kv : count)
    if (c->refs[kv.first] < kv.second) return MINIPIC_ERR_INVALID;
  for (int32_t b : dec) {
    if (--c->refs[b] == 0) {
      c->stamp_of[b] = ++c->stamp;
      c->released.emplace(c->stamp_of[b], b);
    }
  }
  return MINIPIC_OK;
}

}  // extern "C"
