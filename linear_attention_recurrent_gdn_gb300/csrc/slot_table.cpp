// Host slot table: per slot the log length n, the slot whose dense base it
// reads (base_of) and how many other slots index its base (refs).
//
// Rules (DeltaLog page, "Methodology — Base + Log": M-1 append steps, then a
// merge step that rewrites the dense base and clears the log; Flide page,
// "Research method step by step", second step: branches start from their
// request's saved state by indexing it):
//   step      n+1 == M is the merge step: n <- 0, the slot owns its base again;
//             otherwise n <- n+1.  Frozen slots (refs > 0) are refused.
//   fork      dst releases its base, indexes src's base, takes src's n.
//   reset     (set-state / forced merge) release, own base, n <- 0.
// Every operation validates all arguments first and changes nothing on error.
#include <cstdlib>
#include <new>
#include <vector>

#include "../../include/deltalog.h"

struct dl_table {
  int32_t S, M;
  std::vector<int32_t> n, base_of, refs;
  std::vector<uint8_t> mark;   // scratch for duplicate detection
};

extern "C" {

dl_status dl_table_create(int32_t num_slots, int32_t merge_interval, dl_table** out) {
  if (!out) return DL_EINVAL;
  *out = nullptr;
  if (num_slots < 1 || merge_interval < 1) return DL_EINVAL;
  dl_table* t = new (std::nothrow) dl_table;
  if (!t) return DL_ENOMEM;
  try {
    t->S = num_slots;
    t->M = merge_interval;
    t->n.assign(num_slots, 0);
    t->base_of.resize(num_slots);
    for (int32_t s = 0; s < num_slots; ++s) t->base_of[s] = s;
    t->refs.assign(num_slots, 0);
    t->mark.assign(num_slots, 0);
  } catch (...) {
    delete t;
    return DL_ENOMEM;
  }
  *out = t;
  return DL_OK;
}

void dl_table_destroy(dl_table* t) { delete t; }

dl_status dl_table_check(const dl_table* t, const int32_t* slots, int32_t n) {
  if (!t || n < 0 || (n > 0 && !slots)) return DL_EINVAL;
  dl_table* m = const_cast<dl_table*>(t);
  dl_status rc = DL_OK;
  int32_t i = 0;
  for (; i < n; ++i) {
    const int32_t s = slots[i];
    if (s < 0 || s >= t->S || m->mark[s]) {
      rc = DL_EINVAL;
      break;
    }
    m->mark[s] = 1;
  }
  for (int32_t j = 0; j < i; ++j) m->mark[slots[j]] = 0;
  return rc;
}

static bool any_frozen(const dl_table* t, const int32_t* slots, int32_t n) {
  for (int32_t i = 0; i < n; ++i)
    if (t->refs[slots[i]] > 0) return true;
  return false;
}

static void release(dl_table* t, int32_t s) {
  const int32_t b = t->base_of[s];
  if (b != s) {
    t->refs[b] -= 1;
    t->base_of[s] = s;
  }
}

dl_status dl_table_step(dl_table* t, const int32_t* slots, int32_t n, int32_t* plan) {
  dl_status rc = dl_table_check(t, slots, n);
  if (rc != DL_OK) return rc;
  if (any_frozen(t, slots, n)) return DL_EBUSY;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = slots[i];
    const int32_t b = t->base_of[s], len = t->n[s];
    const bool merge = (len + 1 == t->M);
    if (plan) {
      plan[4 * i + 0] = s;
      plan[4 * i + 1] = b;
      plan[4 * i + 2] = len;
      plan[4 * i + 3] = merge ? 1 : 0;
    }
    if (merge) {
      release(t, s);
      t->n[s] = 0;
    } else {
      t->n[s] = len + 1;
    }
  }
  return DL_OK;
}

dl_status dl_table_step_eager(dl_table* t, const int32_t* slots, int32_t n) {
  dl_status rc = dl_table_check(t, slots, n);
  if (rc != DL_OK) return rc;
  if (any_frozen(t, slots, n)) return DL_EBUSY;
  for (int32_t i = 0; i < n; ++i) {
    const int32_t s = slots[i];
    if (t->n[s] != 0 || t->base_of[s] != s) return DL_EINVAL;
  }
  return DL_OK;
}

dl_status dl_table_fork(dl_table* t, int32_t src, const int32_t* dsts, int32_t n) {
  if (!t) return DL_EINVAL;
  if (src < 0 || src >= t->S) return DL_EINVAL;
  dl_status rc = dl_table_check(t, dsts, n);
  if (rc != DL_OK) return rc;
  for (int32_t i = 0; i < n; ++i)
    if (dsts[i] == src) return DL_EINVAL;
  if (any_frozen(t, dsts, n)) return DL_EBUSY;
  const int32_t b = t->base_of[src], len = t->n[src];
  for (int32_t i = 0; i < n; ++i) {
    const int32_t d = dsts[i];
    release(t, d);
    t->base_of[d] = b;
    t->n[d] = len;
    t->refs[b] += 1;
  }
  return DL_OK;
}

dl_status dl_table_reset(dl_table* t, const int32_t* slots, int32_t n) {
  dl_status rc = dl_table_check(t, slots, n);
  if (rc != DL_OK) return rc;
  if (any_frozen(t, slots, n)) return DL_EBUSY;
  for (int32_t i = 0; i < n; ++i) {
    release(t, slots[i]);
    t->n[slots[i]] = 0;
  }
  return DL_OK;
}

// Internal (not in the public header, not exported): set log lengths after a
// checkpoint restore.
__attribute__((visibility("hidden"))) dl_status dl_table_set_n(dl_table* t, const int32_t* slots, int32_t n, const int32_t* len) {
  dl_status rc = dl_table_check(t, slots, n);
  if (rc != DL_OK) return rc;
  for (int32_t i = 0; i < n; ++i)
    if (len[i] < 0 || len[i] >= t->M) return DL_EINVAL;
  for (int32_t i = 0; i < n; ++i) t->n[slots[i]] = len[i];
  return DL_OK;
}

dl_status dl_table_get(const dl_table* t, int32_t* n_log, int32_t* base_of, int32_t* refs) {
  if (!t) return DL_EINVAL;
  for (int32_t s = 0; s < t->S; ++s) {
    if (n_log) n_log[s] = t->n[s];
    if (base_of) base_of[s] = t->base_of[s];
    if (refs) refs[s] = t->refs[s];
  }
  return DL_OK;
}

}  // extern "C"
