// bf16-input, chunk-16 instantiations of the CUDA-core chunked prefill.
#define KDA_SIMT_BF16 1
#define KDA_SIMT_CHUNK 16
#include "prefill_simt.cuh"
