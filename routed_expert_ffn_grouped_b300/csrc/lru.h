// Host LRU core of the expert cache: key -> slot with exact least-recently-used
// replacement and per-batch pinning (pinned slots are never chosen as victims), plus an
// optional usage-pinned hot set: the n_hot most looked-up keys are never evicted.
#pragma once

#include <stdint.h>

#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>

namespace clb {

class LruCore {
  public:
    struct Result {
        int slot;        // slot now holding the key (-1 when result == 2)
        int result;      // 1 resident, 0 inserted, 2 no evictable slot
        int64_t evicted; // key evicted to make room, or -1
    };

    // n_hot: slots reserved for the most used keys (0: plain LRU).
    explicit LruCore(int capacity, int n_hot = 0)
        : key_(capacity, -1), prev_(capacity, -1), next_(capacity, -1), pinned_(capacity, 0), hot_(capacity, 0),
          last_(capacity, 0), n_hot_(n_hot)
    {
        for (int i = capacity - 1; i >= 0; --i)
            free_.push_back(i);
    }

    bool contains(int64_t key) const { return map_.count(key) != 0; }

    // Looks `key` up; a miss inserts it, evicting the least recently used slot that is
    // neither pinned nor hot when the table is full. Either way the key becomes most
    // recently used. A lookup (count_use) adds one use of the key and may move it into
    // the hot set; a prefetch does neither.
    Result access(int64_t key, bool pin, bool count_use = true)
    {
        ++tick_;
        if (count_use)
            ++uses_[key];
        auto it = map_.find(key);
        if (it != map_.end()) {
            const int s = it->second;
            unlink(s);
            push_front(s);
            touch(s);
            if (pin)
                pinned_[s] = 1;
            if (count_use)
                consider_hot(s);
            return {s, 1, -1};
        }
        int s = -1;
        int64_t evicted = -1;
        if (!free_.empty()) {
            s = free_.back();
            free_.pop_back();
        } else {
            for (int v = tail_; v >= 0; v = prev_[v])
                if (!pinned_[v] && !hot_[v]) {
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
        hot_[s] = 0;
        last_[s] = tick_;
        push_front(s);
        if (count_use)
            consider_hot(s);
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
        if (hot_[s])
            hotset_.erase(hot_entry(s));
        map_.erase(it);
        unlink(s);
        key_[s] = -1;
        pinned_[s] = 0;
        hot_[s] = 0;
        free_.push_back(s);
    }

    // Changes the number of hot slots; extra hot keys leave the set (weakest first) and
    // stay resident.
    void set_hot(int n_hot)
    {
        n_hot_ = n_hot < 0 ? 0 : n_hot;
        while ((int)hotset_.size() > n_hot_) {
            const HotEntry weakest = *hotset_.begin();
            hotset_.erase(hotset_.begin());
            hot_[map_.at(std::get<2>(weakest))] = 0;
        }
    }

    int hot_count() const { return (int)hotset_.size(); }
    bool is_hot(int64_t key) const
    {
        auto it = map_.find(key);
        return it != map_.end() && hot_[it->second];
    }

  private:
    // hot keys ordered by (uses, last access, key): the first is the one to demote
    using HotEntry = std::tuple<int64_t, int64_t, int64_t>;

    HotEntry hot_entry(int s) const { return HotEntry(uses_.at(key_[s]), last_[s], key_[s]); }

    // records an access of slot s (its last-access tick; re-files a hot key)
    void touch(int s)
    {
        if (hot_[s]) {
            // the entry was filed under the previous count and tick
            for (auto h = hotset_.begin(); h != hotset_.end(); ++h)
                if (std::get<2>(*h) == key_[s]) {
                    hotset_.erase(h);
                    break;
                }
        }
        last_[s] = tick_;
        if (hot_[s])
            hotset_.insert(hot_entry(s));
    }

    // a resident key with a new use enters the hot set when there is room, or when it has
    // strictly more uses than the weakest hot key, which leaves the set (stays resident)
    void consider_hot(int s)
    {
        if (n_hot_ <= 0 || hot_[s])
            return;
        if ((int)hotset_.size() >= n_hot_) {
            const HotEntry weakest = *hotset_.begin();
            if (uses_.at(key_[s]) <= std::get<0>(weakest))
                return;
            hotset_.erase(hotset_.begin());
            hot_[map_.at(std::get<2>(weakest))] = 0;
        }
        hot_[s] = 1;
        hotset_.insert(hot_entry(s));
    }

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
    std::vector<char> pinned_, hot_;
    std::vector<int64_t> last_;  // tick of each slot's last access
    std::vector<int> free_;
    int head_ = -1, tail_ = -1;
    int n_hot_;
    int64_t tick_ = 0;
    std::unordered_map<int64_t, int64_t> uses_;  // lookups per key, kept across evictions
    std::set<HotEntry> hotset_;
};

}  // namespace clb
