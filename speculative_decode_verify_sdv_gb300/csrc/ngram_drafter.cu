// Host-side n-gram drafter of the speculative-decoding loop: "Stream C --
// Speculative decoding: feasibility verdict + implementation plan", section
// "The delta -- new ENGINE work for greedy n-gram spec-decode": a pure host
// hashtable over the prompt + generated token stream, the last m tokens mapping
// to their most recent continuation.  No device code.
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "sdv.h"

// table[g] = the position right after the latest occurrence of m-gram g that
// has a continuation, i.e. that ends before the last token of the stream.
struct sdv_ngram {
  int m = 0;
  std::vector<int32_t> toks;
  std::unordered_map<std::string, int64_t> table;

  std::string key(size_t end) const {  // the m tokens ending before position `end`
    return std::string(reinterpret_cast<const char*>(toks.data() + end - m), (size_t)m * sizeof(int32_t));
  }
};

namespace {
constexpr int kMaxOrder = 64;
}

extern "C" {

SDV_API sdv_status sdv_ngram_create(int32_t m, sdv_ngram** out) {
  if (out == nullptr) return SDV_ERR_INVALID_ARG;
  *out = nullptr;
  if (m < 1 || m > kMaxOrder) return SDV_ERR_INVALID_ARG;
  sdv_ngram* d = new (std::nothrow) sdv_ngram();
  if (d == nullptr) return SDV_ERR_UNSUPPORTED;
  d->m = m;
  *out = d;
  return SDV_OK;
}

SDV_API sdv_status sdv_ngram_destroy(sdv_ngram* d) {
  delete d;
  return SDV_OK;
}

SDV_API sdv_status sdv_ngram_append(sdv_ngram* d, const int32_t* tokens, int32_t count) {
  if (d == nullptr || count < 0 || (count > 0 && tokens == nullptr)) return SDV_ERR_INVALID_ARG;
  try {
    for (int32_t i = 0; i < count; ++i) {
      const size_t p = d->toks.size();  // index of the new token
      d->toks.push_back(tokens[i]);
      if (p >= (size_t)d->m) d->table[d->key(p)] = (int64_t)p;  // the m-gram ending at p-1 continues at p
    }
  } catch (const std::bad_alloc&) {
    return SDV_ERR_UNSUPPORTED;
  }
  return SDV_OK;
}

SDV_API sdv_status sdv_ngram_propose(const sdv_ngram* d, int32_t k, int32_t* drafts, int32_t* count) {
  if (d == nullptr || count == nullptr || k < 0 || (k > 0 && drafts == nullptr)) return SDV_ERR_INVALID_ARG;
  *count = 0;
  const size_t n = d->toks.size();
  if (k == 0 || n <= (size_t)d->m) return SDV_OK;
  const auto it = d->table.find(d->key(n));
  if (it == d->table.end()) return SDV_OK;
  const size_t c = (size_t)it->second;
  const size_t take = n - c < (size_t)k ? n - c : (size_t)k;
  std::memcpy(drafts, d->toks.data() + c, take * sizeof(int32_t));
  *count = (int32_t)take;
  return SDV_OK;
}

}  // extern "C"
