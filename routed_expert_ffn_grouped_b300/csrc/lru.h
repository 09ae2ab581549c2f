// Host LRU core of the expert cache: key -> slot with exact least-recently-used
// replacement and per-batch pinning (pinned slots are never chosen as victims).
#pragma once

#include <stdint.h>

#include <unordered_map>
#include <vector>

namespace clb {

class LruCore {
  public:
    struct Result {
        int slot;        // slot now holding the key (-1 when result == 2)
        int result;      // 1 resident, 0 inserted, 2 no unpinned slot to evict
        int64_t evicted; // key evicted to make room, or -1
    };

    explicit LruCore(int capacity)
        : key_(capacity, -1), prev_(capacity, -1), next_(capacity, -1), pinned_(capacity, 0)
    {
        for (int i = capacity - 1; i >= 0; --i)
            free_.push_back(i);
    }

    bool contains(int64_t key) const { return map_.count(key) != 0; }

    // Looks `key` up; a miss inserts it, evicting the least recently used unpinned key
    // when the table is full. Either way the key becomes most recently used.
    Result access(int64_t key, bool pin)
    {
        auto it = map_.find(key);
        if (it != map_.end()) {
            const int s = it->second;
            unlink(s);
            push_front(s);
            if (pin)
                pinned_[s] = 1;
            return {s, 1, -1};
        }
        int s = -1;
        int64_t evicted = -1;
        if (!free_.empty()) {
            s = free_.back();
            free_.pop_back();
        } else {
            for (int v = tail_; v >= 0; v = prev_[v])
                if (!pinned_[v]) {
                    s = v;
                    break;
                }
            if (s < 0)
                return {-1, 2, -1};
            evicted = key_[s];
            map_.erase(evicted);
            unlink(s);
        }
        key_[s] = key;
        map_[key] = s;
        pinned_[s] = pin ? 1 : 0;
        push_front(s);
        return {s, 0, evicted};
    }

    void unpin_all()
    {
        for (auto &p : pinned_)
            p = 0;
    }

    // Drops `key` (its slot becomes free).
    void erase(int64_t key)
    {
        auto it = map_.find(key);
        if (it == map_.end())
            return;
        const int s = it->second;
        map_.erase(it);
        unlink(s);
        key_[s] = -1;
        pinned_[s] = 0;
        free_.push_back(s);
    }

  private:
    void unlink(int s)
    {
        if (prev_[s] >= 0)
            next_[prev_[s]] = next_[s];
        else if (head_ == s)
            head_ = next_[s];
        if (next_[s] >= 0)
            prev_[next_[s]] = prev_[s];
        else if (tail_ == s)
            tail_ = prev_[s];
        prev_[s] = next_[s] = -1;
    }

    void push_front(int s)
    {
        prev_[s] = -1;
        next_[s] = head_;
        if (head_ >= 0)
            prev_[head_] = s;
        head_ = s;
        if (tail_ < 0)
            tail_ = s;
    }

    std::unordered_map<int64_t, int> map_;
    std::vector<int64_t> key_;
    std::vector<int> prev_, next_;
    std::vector<char> pinned_;
    std::vector<int> free_;
    int head_ = -1, tail_ = -1;
};

}  // namespace clb
