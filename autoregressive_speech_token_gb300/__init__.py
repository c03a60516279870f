"""Single-stream speech-token decode on GB300: the C-ABI library libsd.so
(CUDA kernels for sm_103a) and its thin Python binding."""

from .sd import (  # noqa: F401
    Decoder, ModelConfig, Sampler, SamplerLadder, SdError, load_library, LIB_PATH, EXPORTS,
    sd_create, sd_load_weights, sd_prefill, sd_step, sd_frame, sd_set_forced_codes, sd_decode_n,
    sd_get_logits, sd_reset, sd_destroy, sd_last_error, sd_get_info,
    sd_qmat_create, sd_qmat_destroy, sd_qmat_dequant, sd_qmat_gemv, sd_qmat_gemm, sd_qmat_gemm16, sd_qmat_gemm_tc, sd_sample_rows, sd_sample_rows_ladder, sd_attend_rows,
    sd_attend_rows_static,
)
