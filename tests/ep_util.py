"""Oracle-backed device steps for the expert-parallel layer's CPU tests (no
method arithmetic: routing, the experts and the combine's rounding are the
oracle's; this file only moves rows)."""
import numpy as np
import torch

from serving_nvfp4_routed_gb300 import synth


def _bf16_tensor(values):
    return torch.from_numpy(np.asarray(values, np.float32)).to(torch.bfloat16)


class OracleOps:
    """The device steps of one rank on the CPU: routing and the experts by
    the oracle (its bank: the rank's experts only), gather and combine by
    index arithmetic, the combine's sum in fp64 and rounded by the oracle."""

    def __init__(self, orc, local_bank):
        self.orc = orc
        self.bank = local_bank

    def route(self, logits, top_k):
        r = self.orc.route(logits.numpy(), top_k)
        return {k: torch.from_numpy(v) for k, v in r.items()}

    def gather(self, x, route, top_k):
        r2s = route["row_to_slot"].numpy()
        offs = route["offsets"].numpy()
        rows = x[torch.from_numpy(r2s // top_k).long()]
        experts = np.searchsorted(offs, np.arange(len(r2s)), side="right") - 1
        return rows.contiguous(), torch.from_numpy(experts.astype(np.int32))

    def experts(self, rows, local_ids, mode, is13=None, is2=None):
        n, d = rows.shape
        if n == 0:
            return torch.empty(0, d, dtype=torch.bfloat16)
        out = self.orc.moe_layer(mode, synth.bf16_bits(rows), local_ids.numpy().reshape(n, 1).astype(np.int32),
                                 np.ones((n, 1), np.float32), self.bank,
                                 is13=None if is13 is None else is13.numpy(),
                                 is2=None if is2 is None else is2.numpy())
        return _bf16_tensor(out)

    def combine(self, y, route, T, top_k):
        yf = y.float().numpy().astype(np.float64)
        s2r = route["slot_to_row"].numpy().reshape(T, top_k)
        w = route["w"].numpy().astype(np.float64)
        acc = np.zeros((T, y.shape[1]))
        for j in range(top_k):
            acc += w[:, j:j + 1] * yf[s2r[:, j]]
        return _bf16_tensor(np.vectorize(self.orc.round_bf16)(acc))


def slice_bank(bank, lo, hi):
    return {k: (v[0][lo:hi], v[1][lo:hi], v[2][lo:hi]) for k, v in bank.items()}
