// lag_list.cuh -- the item list of the one-read column kernels (the GEMM
// operand's columns in quantize.cu, the stored weights' in wquant.cu).
//
// A column's scale needs the maximum over all its rows before any code can
// be written.  The rows are cut into 128-column panels and each panel into
// items of kLagChunk slices; the list holds, for each panel, first its max
// items and, `lag` panels further on, its quantize items, which read the
// same rows again -- from L2, where the max items left them -- once the
// panel's count shows every max item done.  CTAs claim items in list order
// from a counter and work through the items they hold in claim order; a max
// item never waits, and a panel's max items all come before its quantize
// items, so the lowest unfinished item is always being worked on and never
// waits on anything unfinished: every wait ends.
#pragma once

#include <stdint.h>
#include <stdlib.h>

namespace bsg {

constexpr int kLagCols = 128;  // columns per panel
constexpr int kLagChunk = 2;   // slices per item

// Item `it` of the list for P panels of S slices and a lag of L panels.
// (Host-callable too, so that a host test can walk the whole list.)
__host__ __device__ __forceinline__ void lag_item(int64_t it, int64_t P, int64_t S, int64_t L,
                                                  bool &quantize, int64_t &panel,
                                                  int64_t &slice) {
    const int64_t lead = P < L ? P : L;      // panels whose max items come alone
    const int64_t both = P > L ? P - L : 0;  // steps with max and quantize items
    if (it < lead * S) {
        quantize = false;
        panel = it / S;
        slice = it % S;
        return;
    }
    it -= lead * S;
    if (it < both * 2 * S) {
        const int64_t step = L + it / (2 * S), r = it % (2 * S);
        quantize = r >= S;
        panel = quantize ? step - L : step;
        slice = quantize ? r - S : r;
        return;
    }
    it -= both * 2 * S;
    quantize = true;
    panel = both + it / S;
    slice = it % S;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}


// The one-read column quantize's lag, in panels: about 32 MiB of X read
// between a panel's max items and its quantize items.  Measured on a GB300,
// the best lag held 24-32 MiB at every column length (16384 rows: 4 panels,
// 344 us, 2 panels 443 us, 16 panels 418 us; 8192 rows: 8 panels; 4097
// rows: 12-16): shorter lags wait for the max items, longer ones lose the
// tiles from L2 before they are read again.  BSG_COLQ_LAG=1..4096
// overrides it (same results).
inline int64_t colq_lag(int64_t rows) {
    const char *e = getenv("BSG_COLQ_LAG");
    const int v = e ? atoi(e) : 0;
    if (v >= 1 && v <= 4096) return v;
    const int64_t panel_bytes = rows * kLagCols * (int64_t)sizeof(float);
    const int64_t L = (((int64_t)32 << 20) + panel_bytes / 2) / panel_bytes;
    return L < 2 ? 2 : L;
}

}  // namespace bsg
