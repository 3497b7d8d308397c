// status.h - the thread-local message behind tfk_last_error_message(), shared
// by the translation units that implement the C ABI (api.cu, velocity_cache.cpp).
#pragma once

#include "../../include/tfk.h"

namespace tfk {

// Records a printf-style message for tfk_last_error_message() on the calling
// thread and returns `s`.
tfk_status fail(tfk_status s, const char* fmt, ...);

}  // namespace tfk
