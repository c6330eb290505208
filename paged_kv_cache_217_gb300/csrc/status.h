// Per-thread error message and status helpers shared by the host-side code.
#pragma once

#include "paged_kv.h"

namespace pkv {

// Records a printf-style message for pkv_last_error_string() and returns st.
pkv_status_t fail(pkv_status_t st, const char* fmt, ...)
#if defined(__GNUC__)
    __attribute__((format(printf, 2, 3)))
#endif
    ;

// Clears the message and returns PKV_OK.
pkv_status_t ok();

}  // namespace pkv
