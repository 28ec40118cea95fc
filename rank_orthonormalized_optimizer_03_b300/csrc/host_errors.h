// Host-side error reporting shared by the translation units of libdion.so:
// dion_fail() records the detail text that dion_last_error() returns on the
// calling host thread and passes the status code through; dion_ok() clears it.
#pragma once

#include "dion.h"

dion_status_t dion_fail(dion_status_t s, const char* fmt, ...);
dion_status_t dion_ok();
