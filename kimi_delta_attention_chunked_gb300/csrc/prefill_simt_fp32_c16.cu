// fp32-input, chunk-16 instantiations of the CUDA-core chunked prefill.
#define KDA_SIMT_BF16 0
#define KDA_SIMT_CHUNK 16
#include "prefill_simt.cuh"
