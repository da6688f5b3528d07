// Host-side helpers shared by the C-ABI translation units (not part of the public ABI).
#pragma once
#include <string>

#include "../../include/llm.h"

// Record a one-line message for llm_last_error() on this thread and return `s`.
llm_status llm_internal_fail(llm_status s, const std::string& msg);
