/*
 * engram_synth.h -- device twin of the seeded table generator used to make
 * synthetic Engram tables for tests and benchmarks.  This is input generation,
 * not part of the layer: it fills a table of fp8-e4m3 codes and its fp32 block
 * scales exactly as engram_hashed_gram_gb300/synth.py's table_rows() does on
 * the host, so a 98 GB table can be made on the GPU while the host regenerates
 * only the rows it checks.
 *
 * Generator (splitmix64 in counter form, Steele, Lea & Flood, OOPSLA 2014,
 * output mix of Vigna's splitmix64.c):
 *   draw(key, i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15)
 *   mix(z): z = (z ^ z>>30) * 0xBF58476D1CE4E5B9; z = (z ^ z>>27) * 0x94D049BB133111EB;
 *           return z ^ z>>31
 * Row r, channels 4j..4j+3: draw(key_codes, r*head_dim/4 + j); channel 4j+q takes
 * code_qtable[(draw >> 16q) & 0xFFFF].
 * Row r, scale block b: scale_qtable[draw(key_scales, r*nb + b) >> 48],
 * nb = head_dim / scale_block.
 */
#ifndef ENGRAM_SYNTH_H
#define ENGRAM_SYNTH_H

#include <stdint.h>

/* Symbols of the shared library (it is built with hidden default visibility). */
#if defined(__GNUC__)
#define ENGRAM_SYNTH_API __attribute__((visibility("default")))
#else
#define ENGRAM_SYNTH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* engram_synth_stream_t;   /* same type as cudaStream_t */

/* Fills rows [row_begin, row_end) of `table` (device, [R, head_dim] uint8,
 * 16-byte aligned; row r at table + r*head_dim) and of `scale` (device,
 * [R, head_dim/scale_block] fp32; may be NULL to skip the scales).
 * code_qtable (device, 65,536 uint8) and scale_qtable (device, 65,536 fp32) are
 * the quantile tables built on the host.  head_dim must be a multiple of 16.
 * Asynchronous on `stream`.  Returns 0, -1 for a bad argument, -3 for a CUDA
 * error. */
ENGRAM_SYNTH_API int32_t engram_synth_fill_table(uint8_t* table, float* scale, int64_t row_begin, int64_t row_end,
                                int32_t head_dim, int32_t scale_block, uint64_t key_codes,
                                uint64_t key_scales, const uint8_t* code_qtable,
                                const float* scale_qtable, engram_synth_stream_t stream);

/* E8M0 scales of rows [row_begin, row_end): `scale` (device, [R,
 * head_dim/scale_block] uint8) takes e8m0_qtable[draw(key_scales, r*nb + b) >> 48],
 * the same stream positions as the fp32 scales above.  e8m0_qtable: device,
 * 65,536 uint8, built on the host.  Asynchronous on `stream`.  Returns 0, -1
 * for a bad argument, -3 for a CUDA error. */
ENGRAM_SYNTH_API int32_t engram_synth_fill_scales_e8m0(uint8_t* scale, int64_t row_begin, int64_t row_end,
                                                       int32_t head_dim, int32_t scale_block, uint64_t key_scales,
                                                       const uint8_t* e8m0_qtable, engram_synth_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ENGRAM_SYNTH_H */
