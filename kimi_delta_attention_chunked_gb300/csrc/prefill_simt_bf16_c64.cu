// bf16-input, chunk-64 instantiations of the CUDA-core chunked prefill.
#define KDA_SIMT_BF16 1
#define KDA_SIMT_CHUNK 64
#include "prefill_simt.cuh"
