"""GB300 (sm_103a) W4A8 g128 linear layer of QServe's QoQ scheme.

The compute path is ``libqoq.so`` (hand-written CUDA for sm_103a behind the C
ABI of ``include/qoq.h``); ``binding`` is a thin ctypes layer with the same
entry-point names.  PyTorch supplies device memory and the current stream;
every step of the layer runs in the library's kernels.  There is no CPU
fallback: the first call raises if the library is missing.

Names of ``binding`` are re-exported lazily so that ``synth`` (the seeded
input generator) can be imported without loading the CUDA library.
"""
_EXPORTS = (
    "QOQ_ERRORS", "QoQError", "QoQLinear", "build", "library_path", "lib",
    "qoq_gemm_workspace_bytes", "qoq_last_device_status", "qoq_pack_weights",
    "qoq_norm_quant_act", "qoq_packed_weight_bytes", "qoq_quant_act", "qoq_set_debug", "qoq_status_str",
    "qoq_unpack_weights_debug", "qoq_version", "qoq_w4a8_gemm", "qoq_w4a8_gemm_no_alloc", "qoq_no_alloc_last_status",
    "qoq_w4a8_gemm_zero_folded", "qoq_w4ax_act_bytes", "qoq_quant_act_w4ax", "qoq_w4ax_workspace_bytes",
    "qoq_w4ax_gemm", "workspace_for",
)

__all__ = list(_EXPORTS)


def __getattr__(name):
    if name in _EXPORTS:
        from . import binding

        return getattr(binding, name)
    raise AttributeError(name)
