// tmaps.h - TMA tensor maps of the bf16 operands (host side).
#pragma once
#include "plan.h"

// Fill a->maps[] for every MapId; `shadow` is the bf16 parameter copy.
// Returns an mt_status.
int mt_build_tensor_maps(KArgs* a, void* shadow);
