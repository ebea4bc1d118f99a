// The host handle behind the opaque replay_store of the C ABI (library-internal).
#pragma once

#include "launch.h"

struct replay_store {
  replay_config cfg;
  replay_layout lay;
  char* ws;
  rssm::StoreView sv;
  rssm::Shape sh;
  // The ring count every sequence holds, while the host can know it: 0 after an alloc, a
  // full reset, a load or a flush, advanced by each step; -1 (unknown) after a masked reset,
  // a verify or a commit, whose effect depends on device data. Picks kernels only.
  int all_n;
  // Steps alternate between two plan and coefficient buffers (step_parity: the next step's),
  // and a step may start its prep kernel while the previous step's per-head kernel runs when
  // that step is known to have flushed no sequence and ran through the prep (prev_nonflush).
  int step_parity;
  int prev_nonflush;
};

// The step's hint, and the count after a step launched with it.
inline int advance_all_n(const replay_store* st) {
  return st->all_n < 0 ? -1 : (st->all_n + 1 >= st->cfg.window_L ? 0 : st->all_n + 1);
}
