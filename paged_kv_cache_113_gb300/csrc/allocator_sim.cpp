// Allocator policy simulator of libpagedkv.
//
// "The KV Cache Is an Allocator Problem", section "The experiment": one
// deterministic trace of requests (arrival step, prompt, max_new_tokens,
// generated tokens, completion step) replayed against a cache of `capacity`
// token slots under one of three policies:
//   * maximum reservation: one contiguous interval of prompt + max_new_tokens
//     slots, taken at admission;
//   * exact contiguous growth: one contiguous interval of prompt slots at
//     admission, extended in place one slot per generated token, never moved;
//   * paged growth: blocks of B slots on demand, through this library's block
//     manager (floor(capacity / B) blocks handed out 0, 1, 2, ...).
// Step t: every request admitted before t that has not generated all its
// tokens tries to grow by one (trace order); requests whose completion step
// is t release their cache; requests arriving at t are admitted (trace order)
// if their prompt's cache -- for maximum reservation the whole reservation --
// can be allocated. A failed growth drops the request (PK_SIM_DROP) or leaves
// it to try again next step (PK_SIM_STALL). Contiguous placement is first fit.
// Peaks are taken after every successful allocation; one sample per step is
// taken at its end.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <new>
#include <set>
#include <vector>

#include "pagedkv.h"

namespace {

// Free intervals of a contiguous slot range, keyed by start.
class HoleMap {
 public:
  explicit HoleMap(int32_t capacity) {
    if (capacity > 0) holes_[0] = capacity;
  }

  // First fit: the lowest-addressed hole of at least n slots; -1 if none.
  int32_t take(int32_t n) {
    for (auto it = holes_.begin(); it != holes_.end(); ++it) {
      if (it->second < n) continue;
      const int32_t start = it->first, len = it->second;
      holes_.erase(it);
      if (len > n) holes_[start + n] = len - n;
      return start;
    }
    return -1;
  }

  // Takes the single slot at `pos` if it is free.
  bool take_at(int32_t pos) {
    auto it = holes_.find(pos);
    if (it == holes_.end()) return false;
    const int32_t len = it->second;
    holes_.erase(it);
    if (len > 1) holes_[pos + 1] = len - 1;
    return true;
  }

  void give(int32_t start, int32_t n) {
    if (n <= 0) return;
    auto next = holes_.lower_bound(start);
    if (next != holes_.end() && next->first == start + n) {
      n += next->second;
      next = holes_.erase(next);
    }
    if (next != holes_.begin()) {
      auto prev = std::prev(next);
      if (prev->first + prev->second == start) {
        prev->second += n;
        return;
      }
    }
    holes_[start] = n;
  }

  int32_t largest() const {
    int32_t best = 0;
    for (const auto &h : holes_) best = std::max(best, h.second);
    return best;
  }

 private:
  std::map<int32_t, int32_t> holes_;
};

struct Extent {
  int32_t start = 0;
  int32_t len = 0;
};

}  // namespace

extern "C" {

int32_t pk_sim_num_steps(const pk_sim_request *trace, int32_t n) {
  if (n < 0 || (n > 0 && !trace)) return -1;
  int32_t last = 0;
  for (int32_t i = 0; i < n; ++i) last = std::max({last, trace[i].arrival, trace[i].completion});
  return last + 1;
}

pk_status pk_sim_run(const pk_sim_request *trace, int32_t n, int32_t capacity, int32_t policy,
                     int32_t block_size, int32_t rule, pk_sim_summary *summary,
                     pk_sim_sample *samples, int32_t max_samples) {
  if (n < 0 || (n > 0 && !trace) || capacity <= 0 || !summary || max_samples < 0 ||
      (max_samples > 0 && !samples))
    return PK_ERR_INVALID_ARG;
  if (policy != PK_POLICY_MAX_RESERVATION && policy != PK_POLICY_EXACT_CONTIGUOUS &&
      policy != PK_POLICY_PAGED)
    return PK_ERR_INVALID_ARG;
  if (rule != PK_SIM_DROP && rule != PK_SIM_STALL) return PK_ERR_INVALID_ARG;
  if (policy == PK_POLICY_PAGED && (block_size <= 0 || capacity / block_size <= 0))
    return PK_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const pk_sim_request &r = trace[i];
    if (r.arrival < 0 || r.prompt < 1 || r.gen < 0 || r.max_new < r.gen || r.completion <= r.arrival)
      return PK_ERR_INVALID_ARG;
  }
  const int32_t steps = pk_sim_num_steps(trace, n);
  *summary = pk_sim_summary{};
  const bool paged = policy == PK_POLICY_PAGED;
  const bool reserve_max = policy == PK_POLICY_MAX_RESERVATION;
  const int32_t B = paged ? block_size : 1;
  const int32_t num_blocks = paged ? capacity / block_size : 0;
  const int64_t cap = paged ? int64_t(num_blocks) * B : capacity;

  pk_bm *bm = nullptr;
  if (paged) {
    const pk_status st = pk_bm_create(num_blocks, B, nullptr, &bm);
    if (st != PK_OK) return st;
  }
  pk_status result = PK_OK;
  try {
    std::vector<std::vector<int32_t>> arrive(steps), leave(steps);
    for (int32_t i = 0; i < n; ++i) {
      arrive[trace[i].arrival].push_back(i);
      leave[trace[i].completion].push_back(i);
    }
    enum : uint8_t { kWaiting, kActive, kRejected, kDropped, kDone };
    std::vector<uint8_t> state(n, kWaiting);
    std::vector<int32_t> generated(n, 0), admitted_at(n, -1);
    std::vector<Extent> extent(n);
    std::set<int32_t> active;  // trace order
    HoleMap holes(paged ? 0 : capacity);
    // Paged: which blocks are free, kept from the slots the block manager
    // hands out (a slot at offset 0 opens a block) and the blocks a request
    // held when it is released.
    std::vector<uint8_t> is_free(paged ? num_blocks : 0, 1);
    std::vector<std::vector<int32_t>> held(paged ? n : 0);
    std::vector<int64_t> slot_buf;
    int64_t live = 0, reserved = 0;

    auto note_peaks = [&]() {
      summary->peak_live = std::max(summary->peak_live, live);
      summary->peak_reserved = std::max(summary->peak_reserved, reserved);
      summary->peak_waste = std::max(summary->peak_waste, reserved - live);
    };
    auto paged_reserved = [&]() { return int64_t(num_blocks - pk_bm_num_free(bm)) * B; };
    auto release = [&](int32_t i) {
      live -= trace[i].prompt + generated[i];
      if (paged) {
        pk_bm_free_seq(bm, i);
        for (int32_t b : held[i]) is_free[b] = 1;
        held[i].clear();
        reserved = paged_reserved();
      } else {
        holes.give(extent[i].start, extent[i].len);
        reserved -= extent[i].len;
      }
    };
    auto grow = [&](int32_t i) -> bool {
      if (paged) {
        int64_t slot;
        if (pk_bm_append_slots(bm, i, 1, &slot, nullptr, nullptr) != PK_OK) return false;
        if (slot % B == 0) {
          held[i].push_back(int32_t(slot / B));
          is_free[slot / B] = 0;
        }
        reserved = paged_reserved();
        return true;
      }
      if (reserve_max) return true;  // reserved at admission
      if (!holes.take_at(extent[i].start + extent[i].len)) return false;
      extent[i].len += 1;
      reserved += 1;
      return true;
    };
    auto admit = [&](int32_t i) -> bool {
      const pk_sim_request &r = trace[i];
      if (paged) {
        const int64_t need = (int64_t(r.prompt) + B - 1) / B;
        if (need > pk_bm_num_free(bm)) return false;
        slot_buf.resize(size_t(r.prompt));
        if (pk_bm_add_seq(bm, i) != PK_OK ||
            pk_bm_append_slots(bm, i, r.prompt, slot_buf.data(), nullptr, nullptr) != PK_OK)
          return false;
        for (int32_t k = 0; k < r.prompt; k += B) {
          held[i].push_back(int32_t(slot_buf[k] / B));
          is_free[slot_buf[k] / B] = 0;
        }
        reserved = paged_reserved();
        return true;
      }
      const int32_t ask = r.prompt + (reserve_max ? r.max_new : 0);
      const int32_t start = holes.take(ask);
      if (start < 0) return false;
      extent[i] = Extent{start, ask};
      reserved += ask;
      return true;
    };
    auto largest_free = [&]() -> int64_t {
      if (!paged) return holes.largest();
      // Eight flags at a time: an all-held or all-free word needs no byte loop.
      // A run's length is recorded when a held block ends it, and at the end.
      constexpr uint64_t kAllFree = 0x0101010101010101ull;
      int32_t best = 0, run = 0, b = 0;
      auto one = [&](int32_t k) {
        if (is_free[k]) {
          ++run;
        } else {
          best = std::max(best, run);
          run = 0;
        }
      };
      for (; b + 8 <= num_blocks; b += 8) {
        uint64_t w;
        std::memcpy(&w, is_free.data() + b, 8);
        if (w == 0) {
          best = std::max(best, run);
          run = 0;
        } else if (w == kAllFree) {
          run += 8;
        } else {
          for (int32_t k = b; k < b + 8; ++k) one(k);
        }
      }
      for (; b < num_blocks; ++b) one(b);
      return int64_t(std::max(best, run)) * B;
    };

    for (int32_t t = 0; t < steps; ++t) {
      // growth
      for (auto it = active.begin(); it != active.end();) {
        const int32_t i = *it;
        if (admitted_at[i] >= t || generated[i] >= trace[i].gen) {
          ++it;
          continue;
        }
        if (grow(i)) {
          generated[i] += 1;
          live += 1;
          note_peaks();
          ++it;
          continue;
        }
        summary->growth_failures += 1;
        if (cap - reserved >= 1) summary->growth_failures_despite_free += 1;
        if (rule == PK_SIM_DROP) {
          release(i);
          state[i] = kDropped;
          summary->dropped += 1;
          it = active.erase(it);
        } else {
          ++it;
        }
      }
      // completion
      for (int32_t i : leave[t]) {
        if (state[i] != kActive) continue;
        release(i);
        state[i] = kDone;
        active.erase(i);
        summary->completed += 1;
      }
      // admission
      for (int32_t i : arrive[t]) {
        const int64_t free_before = cap - reserved;
        if (admit(i)) {
          state[i] = kActive;
          admitted_at[i] = t;
          active.insert(i);
          live += trace[i].prompt;
          summary->admitted += 1;
          note_peaks();
        } else {
          state[i] = kRejected;
          summary->rejected += 1;
          const int64_t ask = int64_t(trace[i].prompt) + (reserve_max ? trace[i].max_new : 0);
          if (free_before >= ask) summary->rejected_despite_free += 1;
        }
      }
      if (t < max_samples) {
        pk_sim_sample &s = samples[t];
        s.step = t;
        s.active = int32_t(active.size());
        s.live = live;
        s.reserved = reserved;
        s.waste = reserved - live;
        s.free_slots = cap - reserved;
        s.largest_free = largest_free();
      }
    }
    summary->capacity = cap;
    summary->num_steps = steps;
  } catch (const std::bad_alloc &) {
    result = PK_ERR_NOMEM;
  }
  if (bm) pk_bm_destroy(bm);
  return result;
}

}  // extern "C"
