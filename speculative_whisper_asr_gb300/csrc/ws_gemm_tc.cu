// tcgen05 GEMM engine (Blackwell tensor cores, TMEM accumulators, TMA).
#include "ws_internal.cuh"

bool tc_engine_available() { return false; }
