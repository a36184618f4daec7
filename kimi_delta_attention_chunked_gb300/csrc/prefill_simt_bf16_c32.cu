// bf16-input, chunk-32 instantiations of the CUDA-core chunked prefill.
#define KDA_SIMT_BF16 1
#define KDA_SIMT_CHUNK 32
#include "prefill_simt.cuh"
