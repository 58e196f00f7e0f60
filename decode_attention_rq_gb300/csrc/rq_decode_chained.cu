// Chained decode calls that read four to seven residual planes (loop groups of
// five to eight loops, chained anchors: loop l reads every plane from l to the
// anchor).  Same kernels as rq_decode.cu (rq_decode_kernels.cuh), instantiated
// here so that this translation unit compiles beside rq_decode.cu.  One CTA per
// SM: two stages of a unit with up to seven residual planes take most of the
// shared memory (d = 128 with g = 16 and seven planes does not fit: UNSUPPORTED).
#include "rq_decode_kernels.cuh"

namespace rq {
namespace {

template <int D, int GS, bool PAGED>
cudaError_t launch_long(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream) {
  switch (nres) {
    case 4: return launch_t<D, GS, 4, PAGED>(a, num_sms, stream);
    case 5: return launch_t<D, GS, 5, PAGED>(a, num_sms, stream);
    case 6: return launch_t<D, GS, 6, PAGED>(a, num_sms, stream);
    case 7: return launch_t<D, GS, 7, PAGED>(a, num_sms, stream);
  }
  return cudaErrorNotSupported;
}

template <int D, int GS>
cudaError_t launch_long_d(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream) {
  return a.g.paged ? launch_long<D, GS, true>(a, num_sms, nres, stream)
                   : launch_long<D, GS, false>(a, num_sms, nres, stream);
}

}  // namespace

cudaError_t launch_decode_long_chain(const DecodeArgs& a, int num_sms, int nres, cudaStream_t stream) {
  const int d = a.g.d, gs = a.g.g;
  if (d == 128 && gs == 32) return launch_long_d<128, 32>(a, num_sms, nres, stream);
  if (d == 128 && gs == 16) return launch_long_d<128, 16>(a, num_sms, nres, stream);
  if (d == 96 && gs == 32) return launch_long_d<96, 32>(a, num_sms, nres, stream);
  if (d == 96 && gs == 16) return launch_long_d<96, 16>(a, num_sms, nres, stream);
  return cudaErrorNotSupported;
}

}  // namespace rq
