// tmaps.h - TMA tensor maps of the bf16 operands (host side).
#pragma once
#include "plan.h"

// Fill a->maps[] for every MapId; `shadow` is the bf16 parameter copy.
// Returns an mt_status.
int mt_build_tensor_maps(KArgs* a, void* shadow);

// Maps of the single-product test harness: A in MAP_R, B in MAP_WQKV and,
// when C is given, its epilogue map (MAP_E_Y for fp32 C, MAP_E_QKV for bf16).
// a_rpb / b_rpb: rows per box of the operand maps (64, or 128 / 256 for
// K-major operands loaded in taller boxes).
int mt_build_debug_maps(KArgs* a, const void* A, long long a_rows, long long a_cols, const void* B,
                        long long b_rows, long long b_cols, const void* C, long long c_rows, long long c_cols,
                        bool c_f32, int a_rpb, int b_rpb);
