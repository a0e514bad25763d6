// Live-batch former (host): hands out the retained KV cache's slots to
// sessions and turns the set of live sessions into the per-step metadata the
// decode step takes.
//
// quic/efficient-transformers PR #1305 ("Objective"): the retained cache is
// always sized for full_batch_size and a live batch addresses it through
// batch_index.  hw-native-sys/pypto-lib PR #841 (commit message): the live
// batch is the seq_lens descriptor, 1 <= batch <= batch_pad.  antirez/ds4
// PR #530 ("What", the server commits): sessions join and leave between steps
// and every session in plain decode advances in the same batched step.
//
// A session keeps its slot until it is released; a slot never holds two
// sessions.  dsb_batch_form lists the live sessions in slot order (so that the
// metadata of a given set of sessions is the same whatever order they joined
// in), with each one's slot, its KV length after the step (current length +
// tokens_per_seq) and its T pending token ids; dsb_batch_commit then advances
// the lengths.  Sessions are identified by the slot they were given.
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "dsb.h"

struct dsb_batch_former {
  int32_t full_batch_size = 0;
  int32_t ctx = 0;
  std::vector<uint8_t> live;      // per slot
  std::vector<int32_t> length;    // KV rows already written, per slot
  std::vector<int32_t> pending;   // token ids of the next step, per slot (tokens_per_seq each)
  std::vector<uint8_t> has_pending;
  int32_t tps = 1;
};

extern "C" {

dsb_status dsb_batch_former_create(int full_batch_size, int ctx, int tokens_per_seq, dsb_batch_former** out) {
  if (!out) return DSB_ERR_INVALID_ARG;
  *out = nullptr;
  if (full_batch_size < 1 || full_batch_size > DSB_MAX_SEQS || ctx < 1 || tokens_per_seq < 1 ||
      tokens_per_seq > ctx || (long long)full_batch_size * tokens_per_seq > DSB_MAX_TOKENS)
    return DSB_ERR_INVALID_ARG;
  dsb_batch_former* b = new (std::nothrow) dsb_batch_former();
  if (!b) return DSB_ERR_INVALID_ARG;
  b->full_batch_size = full_batch_size;
  b->ctx = ctx;
  b->tps = tokens_per_seq;
  b->live.assign((size_t)full_batch_size, 0);
  b->length.assign((size_t)full_batch_size, 0);
  b->pending.assign((size_t)full_batch_size * tokens_per_seq, 0);
  b->has_pending.assign((size_t)full_batch_size, 0);
  *out = b;
  return DSB_OK;
}

void dsb_batch_former_destroy(dsb_batch_former* b) { delete b; }

dsb_status dsb_batch_join(dsb_batch_former* b, int prefill_length, int32_t* slot_out) {
  if (!b || !slot_out) return DSB_ERR_INVALID_ARG;
  if (prefill_length < 0 || prefill_length > b->ctx) return DSB_ERR_INVALID_ARG;
  for (int s = 0; s < b->full_batch_size; ++s) {
    if (!b->live[(size_t)s]) {
      b->live[(size_t)s] = 1;
      b->length[(size_t)s] = prefill_length;
      b->has_pending[(size_t)s] = 0;
      *slot_out = s;
      return DSB_OK;
    }
  }
  return DSB_ERR_UNSUPPORTED;  // every slot is taken
}

dsb_status dsb_batch_leave(dsb_batch_former* b, int slot) {
  if (!b || slot < 0 || slot >= b->full_batch_size || !b->live[(size_t)slot]) return DSB_ERR_INVALID_ARG;
  b->live[(size_t)slot] = 0;
  b->has_pending[(size_t)slot] = 0;
  b->length[(size_t)slot] = 0;
  return DSB_OK;
}

dsb_status dsb_batch_submit(dsb_batch_former* b, int slot, const int32_t* token_ids) {
  if (!b || !token_ids || slot < 0 || slot >= b->full_batch_size || !b->live[(size_t)slot]) return DSB_ERR_INVALID_ARG;
  if (b->length[(size_t)slot] + b->tps > b->ctx) return DSB_ERR_UNSUPPORTED;  // the cache row would overflow
  std::memcpy(&b->pending[(size_t)slot * b->tps], token_ids, sizeof(int32_t) * (size_t)b->tps);
  b->has_pending[(size_t)slot] = 1;
  return DSB_OK;
}

dsb_status dsb_batch_form(const dsb_batch_former* b, int32_t* batch_index, int32_t* seq_lens, int32_t* token_ids,
                          int32_t* n_seq_out) {
  if (!b || !batch_index || !seq_lens || !token_ids || !n_seq_out) return DSB_ERR_INVALID_ARG;
  int n = 0;
  for (int s = 0; s < b->full_batch_size; ++s) {
    if (!b->live[(size_t)s] || !b->has_pending[(size_t)s]) continue;
    batch_index[n] = s;
    seq_lens[n] = b->length[(size_t)s] + b->tps;
    std::memcpy(&token_ids[(size_t)n * b->tps], &b->pending[(size_t)s * b->tps], sizeof(int32_t) * (size_t)b->tps);
    ++n;
  }
  *n_seq_out = n;
  return DSB_OK;
}

dsb_status dsb_batch_commit(dsb_batch_former* b, const int32_t* batch_index, int n_seq) {
  if (!b || (n_seq > 0 && !batch_index) || n_seq < 0 || n_seq > b->full_batch_size) return DSB_ERR_INVALID_ARG;
  for (int i = 0; i < n_seq; ++i) {
    const int s = batch_index[i];
    if (s < 0 || s >= b->full_batch_size || !b->live[(size_t)s] || !b->has_pending[(size_t)s])
      return DSB_ERR_INVALID_ARG;
  }
  for (int i = 0; i < n_seq; ++i) {
    const int s = batch_index[i];
    b->length[(size_t)s] += b->tps;
    b->has_pending[(size_t)s] = 0;
  }
  return DSB_OK;
}

int dsb_batch_length(const dsb_batch_former* b, int slot) {
  if (!b || slot < 0 || slot >= b->full_batch_size || !b->live[(size_t)slot]) return -1;
  return b->length[(size_t)slot];
}

}  // extern "C"
