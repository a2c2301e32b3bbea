"""Python binding of ``libllm.so``, the sm_103a Llama decoder forward pass.

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels behind the C ABI declared in ``include/llm.h``.  The functions keep
the C names.  PyTorch provides device memory and streams; tensors are passed
by ``data_ptr()``.  Importing this module raises ImportError when the library
has not been built — there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libllm.so")

LLM_OK, LLM_NO_KV_ROOM, LLM_ERR_INVALID, LLM_ERR_ALLOC, LLM_ERR_COMPUTE = 0, 1, -1, -2, -3
LLM_BATCH_TOKENS_ON_DEVICE = 1
LLM_WTYPE_Q8_0 = 1

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with llama_decoder_forward_02_gb300.build.build()")

_lib = ctypes.CDLL(LIB_PATH)

c_i32, c_i64, c_f32, c_vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p
c_i32p = ctypes.POINTER(ctypes.c_int32)
c_i8p = ctypes.POINTER(ctypes.c_int8)


class llm_hparams(ctypes.Structure):
    _fields_ = [("n_vocab", c_i32), ("n_embd", c_i32), ("n_layer", c_i32), ("n_head", c_i32),
                ("n_head_kv", c_i32), ("head_dim", c_i32), ("n_ff", c_i32),
                ("rms_eps", c_f32), ("rope_theta", c_f32), ("tied_output", c_i32)]


class llm_weights(ctypes.Structure):
    _fields_ = [("token_embd", c_vp), ("output_norm", c_vp), ("output", c_vp),
                ("attn_norm", ctypes.POINTER(c_vp)), ("wq", ctypes.POINTER(c_vp)),
                ("wk", ctypes.POINTER(c_vp)), ("wv", ctypes.POINTER(c_vp)), ("wo", ctypes.POINTER(c_vp)),
                ("ffn_norm", ctypes.POINTER(c_vp)), ("w_gate", ctypes.POINTER(c_vp)),
                ("w_up", ctypes.POINTER(c_vp)), ("w_down", ctypes.POINTER(c_vp))]


class llm_batch(ctypes.Structure):
    _fields_ = [("n_tokens", c_i32), ("token", c_i32p), ("pos", c_i32p), ("seq_id", c_i32p),
                ("output", c_i8p), ("flags", c_i32)]


class llm_sampling(ctypes.Structure):
    _fields_ = [("temperature", c_f32), ("top_k", c_i32), ("top_p", c_f32), ("min_p", c_f32),
                ("repeat_penalty", c_f32), ("penalty_last_n", c_i32)]


def _proto(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_model_p = ctypes.POINTER(c_vp)
llm_model_create = _proto("llm_model_create", c_i32, ctypes.POINTER(llm_hparams), ctypes.POINTER(llm_weights),
                          c_vp, ctypes.POINTER(c_vp))
llm_model_free = _proto("llm_model_free", None, c_vp)
llm_model_quantize = _proto("llm_model_quantize", c_i32, c_vp, c_i32, c_vp)
llm_kv_alloc = _proto("llm_kv_alloc", c_i32, c_vp, c_i32, c_i32, c_i32, c_vp, ctypes.POINTER(c_vp))
llm_kv_free = _proto("llm_kv_free", None, c_vp)
llm_decode = _proto("llm_decode", c_i32, c_vp, ctypes.POINTER(llm_batch))
llm_get_logits = _proto("llm_get_logits", c_vp, c_vp, c_i32p)
llm_get_logits_ith = _proto("llm_get_logits_ith", c_vp, c_vp, c_i32)
llm_get_argmax = _proto("llm_get_argmax", c_i32, c_vp, c_i32p, c_i32)
llm_generate = _proto("llm_generate", c_i32, c_vp, c_i32, c_i32, c_vp)
llm_sample = _proto("llm_sample", c_i32, c_vp, ctypes.POINTER(llm_sampling), ctypes.POINTER(c_f32), c_i32p, c_i32,
                    c_i32p, c_i32)
llm_op_sample = _proto("llm_op_sample", c_i32, c_vp, c_i32, c_i32, ctypes.POINTER(llm_sampling), c_vp, c_vp, c_i32,
                       c_vp, c_vp)
llm_seq_pos_max = _proto("llm_seq_pos_max", c_i32, c_vp, c_i32)
llm_seq_clear = _proto("llm_seq_clear", c_i32, c_vp, c_i32)
llm_seq_shift = _proto("llm_seq_shift", c_i32, c_vp, c_i32, c_i32, c_i32)
llm_synchronize = _proto("llm_synchronize", c_i32, c_vp)
llm_last_error = _proto("llm_last_error", ctypes.c_char_p, c_vp)
llm_debug_hidden = _proto("llm_debug_hidden", c_i32, c_vp, c_vp, c_i32, c_i32)
llm_debug_fail_alloc = _proto("llm_debug_fail_alloc", c_i32, c_i32)
llm_set_option = _proto("llm_set_option", c_i32, c_vp, ctypes.c_char_p, c_i32)
llm_kernel_launches = _proto("llm_kernel_launches", c_i64, c_vp)
llm_kernel_timing = _proto("llm_kernel_timing", c_i32, c_vp, c_i32)
llm_kernel_time = _proto("llm_kernel_time", c_i32, c_vp, c_i32, ctypes.POINTER(ctypes.c_double),
                         ctypes.POINTER(c_i64), ctypes.POINTER(ctypes.c_char_p))
llm_batch_check = _proto("llm_batch_check", c_i32, c_i32, c_i32, c_i32, c_i32, c_i32p, ctypes.POINTER(llm_batch),
                         c_i32p, c_i32p, c_i32p, c_i32p)
llm_op_gemv = _proto("llm_op_gemv", c_i32, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_i64, c_vp)
llm_op_gemm = _proto("llm_op_gemm", c_i32, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp)
llm_op_quantize_q8_0 = _proto("llm_op_quantize_q8_0", c_i32, c_vp, c_i32, c_i32, c_vp, c_vp)
llm_op_gemv_q8_0 = _proto("llm_op_gemv_q8_0", c_i32, c_vp, c_vp, c_vp, c_i32, c_i32, c_vp)
llm_op_wait_check = _proto("llm_op_wait_check", c_i32, c_i32, c_i32, c_vp, c_vp)
llm_op_attn_decode_scratch_bytes = _proto("llm_op_attn_decode_scratch_bytes", c_i64, c_i32, c_i32, c_i32, c_i32)
llm_op_attn_decode = _proto("llm_op_attn_decode", c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32,
                            c_i32, c_i32, c_i32, c_i32, c_vp, c_i64, c_vp)
llm_op_attn_decode_noalloc = _proto("llm_op_attn_decode_noalloc", c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32,
                                    c_i32, c_i32, c_i32, c_i32, c_i32, c_i32, c_vp)
llm_op_attn_prefill = _proto("llm_op_attn_prefill", c_i32, c_vp, c_vp, c_vp, c_i32p, c_i32p, c_vp, c_i32, c_i32,
                             c_i32, c_i32, c_i32, c_i32, c_vp)

EXPORTED = [n for n in dir() if n.startswith("llm_") and callable(globals()[n]) and
            not isinstance(globals()[n], type)]


class LlmError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{msg} (code {code})")
        self.code = code


def check(code, handle=None):
    if code < 0:
        raise LlmError(code, llm_last_error(handle).decode())
    return code


# ---------------------------------------------------------------- marshalling helpers

def hparams(shape) -> llm_hparams:
    """llm_hparams from any object with the Llama hyper-parameter fields."""
    return llm_hparams(shape.n_vocab, shape.n_embd, shape.n_layer, shape.n_head, shape.n_head_kv,
                       shape.head_dim, shape.n_ff, shape.rms_eps, shape.rope_theta, int(bool(shape.tied_output)))


def weights(tensors: dict, n_layer: int, tied: bool):
    """llm_weights from device tensors named by their GGUF tags.  Returns the
    struct and the pointer arrays it references (keep both alive)."""
    arr = {}
    keep = []
    for leaf, field in (("attn_norm", "attn_norm"), ("attn_q", "wq"), ("attn_k", "wk"), ("attn_v", "wv"),
                        ("attn_output", "wo"), ("ffn_norm", "ffn_norm"), ("ffn_gate", "w_gate"),
                        ("ffn_up", "w_up"), ("ffn_down", "w_down")):
        a = (c_vp * n_layer)(*[tensors[f"blk.{i}.{leaf}"].data_ptr() for i in range(n_layer)])
        keep.append(a)
        arr[field] = ctypes.cast(a, ctypes.POINTER(c_vp))
    w = llm_weights(tensors["token_embd"].data_ptr(), tensors["output_norm"].data_ptr(),
                    None if tied else tensors["output"].data_ptr(), **arr)
    return w, keep


def _arr(ctype, values):
    if values is None:
        return None, None
    a = (ctype * len(values))(*[int(v) for v in values])
    return ctypes.cast(a, ctypes.POINTER(ctype)), a


def batch(tokens=None, pos=None, seq_id=None, output=None, n_tokens=None, token_dev_ptr=None):
    """llm_batch from host sequences (or a device token pointer).  Returns the
    struct and the arrays it references (keep both alive)."""
    keep = []
    if token_dev_ptr is not None:
        tok_p = ctypes.cast(c_vp(token_dev_ptr), c_i32p)
        n = int(n_tokens)
        flags = LLM_BATCH_TOKENS_ON_DEVICE
    else:
        tok_p, a = _arr(ctypes.c_int32, tokens)
        keep.append(a)
        n = len(tokens) if n_tokens is None else int(n_tokens)
        flags = 0
    pos_p, a = _arr(ctypes.c_int32, pos); keep.append(a)
    seq_p, a = _arr(ctypes.c_int32, seq_id); keep.append(a)
    out_p, a = _arr(ctypes.c_int8, output); keep.append(a)
    return llm_batch(n, tok_p, pos_p, seq_p, out_p, flags), keep


class _DeviceArray:
    """A raw device pointer exposed through __cuda_array_interface__."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (int(ptr), False),
                                         "version": 2, "strides": None}


def device_view(ptr, shape, typestr="<f4"):
    """Zero-copy torch view of library-owned device memory (e.g. the logits)."""
    import torch
    return torch.as_tensor(_DeviceArray(ptr, shape, typestr), device="cuda")


def logits_numpy(ctx, n_vocab):
    """Copy of the last decode's logits [n_outputs][n_vocab] as float64 numpy."""
    import numpy as np
    ctx.synchronize()
    p, n = ctx.logits_ptr()
    if n == 0 or not p:
        return np.zeros((0, n_vocab))
    return device_view(p, (n, n_vocab)).cpu().double().numpy()


class Model:
    """Owns an llm_model handle."""

    def __init__(self, shape, tensors: dict, stream=0):
        self.shape = shape
        w, keep = weights(tensors, shape.n_layer, bool(shape.tied_output))
        hp = hparams(shape)
        h = c_vp()
        check(llm_model_create(ctypes.byref(hp), ctypes.byref(w), c_vp(stream), ctypes.byref(h)))
        self.handle = h

    def quantize(self, wtype=None, stream=0):
        """llm_model_quantize (default LLM_WTYPE_Q8_0)."""
        check(llm_model_quantize(self.handle, LLM_WTYPE_Q8_0 if wtype is None else wtype, c_vp(stream)))

    def free(self):
        if self.handle:
            llm_model_free(self.handle)
            self.handle = None


class Context:
    """Owns an llm_ctx handle; methods marshal to the C calls of the same name."""

    def __init__(self, model: Model, n_ctx: int, n_seq_max: int = 1, n_ubatch: int = 512, stream=0):
        self.model = model
        h = c_vp()
        check(llm_kv_alloc(model.handle, n_ctx, n_seq_max, n_ubatch, c_vp(stream), ctypes.byref(h)))
        self.handle = h

    def decode(self, tokens=None, pos=None, seq_id=None, output=None, token_dev_ptr=None, n_tokens=None):
        b, keep = batch(tokens, pos, seq_id, output, n_tokens=n_tokens, token_dev_ptr=token_dev_ptr)
        rc = llm_decode(self.handle, ctypes.byref(b))
        return check(rc, self.handle)

    def logits_ptr(self):
        n = ctypes.c_int32(0)
        p = llm_get_logits(self.handle, ctypes.byref(n))
        return p, n.value

    def logits_ith_ptr(self, i):
        return llm_get_logits_ith(self.handle, i)

    def argmax(self, capacity=1 << 16):
        out = (ctypes.c_int32 * capacity)()
        n = check(llm_get_argmax(self.handle, out, capacity), self.handle)
        return list(out[:n])

    def sample(self, params: llm_sampling, u=None, history=()):
        """Tokens the sampling chain picks for the output rows of the last decode
        (u: one uniform in [0, 1) per output row; history: earlier tokens)."""
        n = self.n_outputs()
        ua = (c_f32 * max(n, 1))(*(u if u is not None else [0.0] * n))
        h = list(history)
        ha = (c_i32 * max(len(h), 1))(*h)
        out = (c_i32 * max(n, 1))()
        rc = check(llm_sample(self.handle, ctypes.byref(params), ua, ha, len(h), out, max(n, 1)), self.handle)
        return list(out)[:rc]

    def n_outputs(self):
        n = ctypes.c_int32(0)
        llm_get_logits(self.handle, ctypes.byref(n))
        return n.value

    def generate(self, seq_id, n_steps, tokens_out_ptr):
        return check(llm_generate(self.handle, seq_id, n_steps, c_vp(tokens_out_ptr)), self.handle)

    def seq_pos_max(self, s):
        return llm_seq_pos_max(self.handle, s)

    def seq_clear(self, s):
        return check(llm_seq_clear(self.handle, s), self.handle)

    def seq_shift(self, s, p0, n_discard):
        """Drop positions [p0, p0 + n_discard) of sequence s and shift the rest down."""
        return check(llm_seq_shift(self.handle, s, p0, n_discard), self.handle)

    def synchronize(self):
        return check(llm_synchronize(self.handle), self.handle)

    def set_option(self, key, value):
        return check(llm_set_option(self.handle, key.encode(), int(value)), self.handle)

    def debug_hidden(self, ptr, max_rows, max_ubatches):
        return check(llm_debug_hidden(self.handle, c_vp(ptr) if ptr else None, max_rows, max_ubatches), self.handle)

    def kernel_launches(self):
        return llm_kernel_launches(self.handle)

    def kernel_timing(self, enable):
        return check(llm_kernel_timing(self.handle, int(enable)), self.handle)

    def kernel_times(self):
        """{kernel class name: (total ms, launches)} since timing was enabled."""
        out = {}
        k = 0
        while True:
            ms, n, name = ctypes.c_double(), c_i64(), ctypes.c_char_p()
            if llm_kernel_time(self.handle, k, ctypes.byref(ms), ctypes.byref(n), ctypes.byref(name)) != 0:
                break
            if n.value:
                out[name.value.decode()] = (ms.value, n.value)
            k += 1
        return out

    def last_error(self):
        return llm_last_error(self.handle).decode()

    def free(self):
        if self.handle:
            llm_kv_free(self.handle)
            self.handle = None
