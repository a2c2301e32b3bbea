"""Helpers for end-to-end GPU parity tests: the same synthetic weights go to
the CUDA library (device tensors, through the C ABI) and to the oracle
(host bf16 bit arrays)."""
import numpy as np
import torch

import synth
from oracle import llama as O

# Tolerances of the parity bar (logits of unit order).
LOGIT_TOL = 5e-2
HIDDEN_REL_TOL = 1e-2

# Medium shapes that exercise ragged tiles and every head_dim quickly.
MED64 = synth.Shape(n_vocab=1024, n_embd=256, n_layer=3, n_head=4, n_head_kv=2, head_dim=64, n_ff=700,
                    rms_eps=1e-5, rope_theta=10000.0, tied_output=False)
MED128 = synth.Shape(n_vocab=2048, n_embd=512, n_layer=2, n_head=4, n_head_kv=1, head_dim=128, n_ff=1000,
                     rms_eps=1e-5, rope_theta=500000.0, tied_output=True)


class Pair:
    def __init__(self, lib, shape, seed, n_ctx, n_seq=1, n_ubatch=512, dtype=np.float64, device_draw=False,
                 q8=False):
        """q8: the library model is re-encoded as Q8_0 (llm_model_quantize) and
        the oracle model is its own Q8_0 model (Model.quantized_q8_0)."""
        self.lib, self.shape = lib, shape
        t = synth.make_weights(shape, seed, "cuda" if device_draw else "cpu")
        self.dev = {k: v.cuda() for k, v in t.items()}
        host = synth.host_weights(t)
        del t
        st = torch.cuda.current_stream().cuda_stream
        self.model = lib.Model(shape, self.dev, stream=st)
        if q8:
            self.model.quantize(stream=st)
        self.ctx = lib.Context(self.model, n_ctx, n_seq, n_ubatch, stream=st)
        self.dev = None        # the library copied what it needs
        torch.cuda.empty_cache()
        self.om = O.Model(O.Hparams.of(shape), host, dtype)
        if q8:
            self.om = self.om.quantized_q8_0()
        self.oc = O.Context(self.om, n_ctx, n_seq, n_ubatch)

    def logits(self):
        self.ctx.synchronize()
        return self.lib.logits_numpy(self.ctx, self.shape.n_vocab)

    def free(self):
        self.ctx.free()
        self.model.free()


def compare_logits(got, ref, tol=LOGIT_TOL):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    assert err <= tol, f"max |dlogit| = {err}"
    return err


def top1_agreement(got, ref, margin=0.1):
    """Fraction of rows with the oracle's top-2 margin > margin whose argmax agrees."""
    srt = np.sort(ref, axis=1)
    m = srt[:, -1] - srt[:, -2] > margin
    if not m.any():
        return 1.0, 0
    agree = np.argmax(got[m], axis=1) == np.argmax(ref[m], axis=1)
    return float(agree.mean()), int(m.sum())
