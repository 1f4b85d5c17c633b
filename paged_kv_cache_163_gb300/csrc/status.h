// Status helpers shared by the host and device translation units.
#pragma once

#include "pkv.h"

namespace pkv {

// Record a one-line reason for the calling thread and return `s`.
pkv_status fail(pkv_status s, const char *reason);

}  // namespace pkv
