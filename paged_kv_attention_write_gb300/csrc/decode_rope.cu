// decode_rope.cu -- the decode instantiations that rotate the query (RoPE, GPT-J pairs)
// at position context_len - 1 and apply the position-dependent query scale before the
// scores (TensorSharp "Mistral 3" page, section 4.2).  A translation unit of its own so
// that the plain kernels keep their code and both compile in parallel.
#include "decode_kernels.cuh"

namespace pa {

int dispatch_decode_rope(const DecodeParams &prm, pa_dtype kv_dtype, int D, int G, const CUtensorMap &km,
                         const CUtensorMap &vm, cudaStream_t st) {
    return dispatch_kv<true>(prm, kv_dtype, D, G, km, vm, st);
}

}  // namespace pa
