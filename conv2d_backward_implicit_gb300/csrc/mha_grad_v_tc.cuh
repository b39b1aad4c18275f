// mha_grad_v_tc.cuh -- tensor-core kernel of the attention dV (included by
// mha_grad_v.cu).
namespace mhadv {
namespace {

bool tc_applies(const void *, const void *, const void *, const mha_grad_v_params *, int) { return false; }

int launch_tc(const void *, const void *, const void *, const float *, float *, const mha_grad_v_params *, int,
              cudaStream_t) {
    return DGRAD_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace mhadv
