// prefill.cu -- varlen causal prefill on the paged pools (tcgen05 / TMEM).
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

cudaError_t launch_prefill(const PrefillParams &p, const pkv_cache_desc &cache,
                           const CUtensorMap *tmap_q, const CUtensorMap *tmap_k,
                           const CUtensorMap *tmap_v, cudaStream_t stream) {
    (void)p; (void)cache; (void)tmap_q; (void)tmap_k; (void)tmap_v; (void)stream;
    return cudaErrorNotSupported;
}

}  // namespace pkv
