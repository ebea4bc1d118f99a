// The host handle behind the opaque replay_store of the C ABI (library-internal).
#pragma once

#include "launch.h"

struct replay_store {
  replay_config cfg;
  replay_layout lay;
  char* ws;
  rssm::StoreView sv;
  rssm::Shape sh;
};
