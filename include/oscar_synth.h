/*
 * oscar_synth.h -- C ABI of liboscar_synth: the seeded synthetic-input
 * generator on the GPU.  It draws the same numbers as
 * int2_kv_cache_02_gb300/synth.py (the test and benchmark inputs); it is not
 * part of the OScaR method and holds none of its arithmetic.
 *
 * Definition: splitmix64 used as a counter-based generator (Steele, Lea &
 * Flood, OOPSLA 2014): output n of stream `seed` is
 * mix(seed + (n+1) * 0x9E3779B97F4A7C15).  Element counter
 * e = ((b*H + h) * 2^32 + t) * 128 + c takes outputs 3e, 3e+1, 3e+2, whose
 * twelve 16-bit fields sum (minus 6*65536) to an Irwin-Hall integer; times
 * 2^-16 in fp32, times the channel factor, times the token factor (fp32,
 * round to nearest even each), rounded to bf16.
 */
#ifndef OSCAR_SYNTH_H
#define OSCAR_SYNTH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Fills out[((b*H + h)*out_T + t)*128 + c] for b < nB, h < H, t < n_t with
 * element (b0 + b, h, t0 + t, c) of the logical [*][H][*][128] tensor.
 *  chan_factor  device fp32 [128] or NULL (all 1)
 *  tok_factor   device fp32 [nB][n_t] or NULL (all 1)
 * All pointers device memory, `out` 16-byte aligned.  Asynchronous on
 * `stream`.  Returns 0 on success, 1 on a bad argument, 2 on a CUDA error.
 */
int oscar_synth_bf16(uint16_t* out, int nB, int H, int b0, int out_T, int t0, int n_t,
                     unsigned long long seed, const float* chan_factor, const float* tok_factor,
                     void* stream);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_SYNTH_H */
