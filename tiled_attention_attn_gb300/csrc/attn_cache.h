// A bounded least-recently-used cache of per-shape schedules, independent of
// CUDA so that its eviction policy can be exercised on the host alone.
//
// An entry that a stream capture has referenced is pinned: a captured graph
// keeps reading its device copy at every replay, so it is never evicted.
// Other entries beyond the capacity are evicted least recently used first and
// handed to the release callback, which frees their device memory in stream
// order after their last use.  Eviction is skipped while the calling stream
// captures (its stream operations would become part of the graph); the
// cache then runs over capacity until the next call outside a capture.
#pragma once
#include <cstddef>
#include <cstdint>
#include <functional>
#include <map>
#include <memory>

namespace attn {

template <class Key, class Entry>
class LruCache {
 public:
  explicit LruCache(size_t capacity) : cap_(capacity) {}

  Entry* find(const Key& k) {
    auto it = map_.find(k);
    if (it == map_.end()) return nullptr;
    it->second->lru = ++tick_;
    return it->second.get();
  }

  // Inserts a new entry (the key must be absent), evicting first when full
  // and allowed.  Returns the stored entry.
  Entry* insert(const Key& k, std::unique_ptr<Entry> e, bool may_evict,
                const std::function<void(Entry&)>& release) {
    if (may_evict) trim(cap_ == 0 ? 0 : cap_ - 1, release);
    e->lru = ++tick_;
    Entry* p = e.get();
    map_.emplace(k, std::move(e));
    return p;
  }

  // Evicts unpinned entries, least recently used first, until at most `n`
  // entries remain or only pinned ones are left.
  void trim(size_t n, const std::function<void(Entry&)>& release) {
    while (map_.size() > n) {
      auto victim = map_.end();
      for (auto it = map_.begin(); it != map_.end(); ++it)
        if (!it->second->pinned && (victim == map_.end() || it->second->lru < victim->second->lru)) victim = it;
      if (victim == map_.end()) return;
      release(*victim->second);
      map_.erase(victim);
    }
  }

  size_t size() const { return map_.size(); }
  size_t capacity() const { return cap_; }
  template <class F>
  void for_each(F f) {
    for (auto& kv : map_) f(*kv.second);
  }

 private:
  size_t cap_;
  uint64_t tick_ = 0;
  std::map<Key, std::unique_ptr<Entry>> map_;
};

}  // namespace attn
