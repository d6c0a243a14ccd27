// internal.h -- declarations shared by the library's translation units; not
// part of the C ABI (include/kda.h) and not exported.
#pragma once

// kda_linear with an optional programmatic-dependent launch (the kernel may
// start while the previous kernel on the stream finishes; it waits for that
// kernel's results before reading x). Same arguments and return codes as
// kda_linear.
__attribute__((visibility("hidden"))) int kda_linear_enqueue(const void* x, long long rows, long long ldx,
                                                             const void* w, long long N, long long K, void* y,
                                                             long long ldy, void* cuda_stream, bool pdl);
