// The fused INT2 decode for query groups of 3, 5..7 and 9..16 heads per KV
// head: the kernels of decode_int2.cu instantiated with padding heads (and
// slices of 8 heads above 8), in a translation unit of their own so that the
// two build in parallel.
#define OSCAR_DECODE_PAD_TU
#include "decode_int2.cu"
