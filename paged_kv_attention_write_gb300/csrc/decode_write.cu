// decode_write.cu -- the decode instantiations that first write each sequence's new token
// into its cache slot (pa_reshape_and_cache of one token per sequence, TensorSharp "Mistral 3"
// page, section 11: K/V scatter through slotMapping, then the per-sequence paged attention)
// in the same launch.  A translation unit of its own so that the plain kernels keep their code
// and all compile in parallel.
#include "decode_kernels.cuh"

namespace pa {

int dispatch_decode_write(const DecodeParams &prm, pa_dtype kv_dtype, int D, int G, const CUtensorMap &km,
                          const CUtensorMap &vm, cudaStream_t st) {
    return dispatch_kv<false, true>(prm, kv_dtype, D, G, km, vm, st);
}

}  // namespace pa
