"""Device buffers with canaries, for the GPU parity tests.

Every buffer is laid out as [lead words][payload words][1024 canary words]:
the 4 KB of canary words past the end (and any lead words before a shifted
start) must come back bit-identical after a kernel ran.
"""
import numpy as np
import torch

from masking_tm_affine_gb300 import synth

CANARY = int(synth.CANARY_U32)
CANARY_WORDS = 1024  # 4 KB past every tensor end


class DevBuf:
    def __init__(self, payload, lead: int = 0, device="cuda"):
        payload = np.ascontiguousarray(payload).reshape(-1)
        if payload.dtype.itemsize != 4:
            raise TypeError("32-bit payload expected")
        self.n = payload.size
        self.lead = lead
        words = np.full(lead + self.n + CANARY_WORDS, CANARY, dtype=np.uint32)
        words[lead:lead + self.n] = payload.view(np.uint32)
        self.t = torch.from_numpy(words.view(np.float32)).to(device)
        self.ptr = self.t.data_ptr() + 4 * lead

    @classmethod
    def empty(cls, n: int, lead: int = 0, fill=CANARY):
        return cls(np.full(n, fill, dtype=np.uint32), lead)

    def words(self) -> np.ndarray:
        return self.t.cpu().numpy().view(np.uint32)

    def payload_u32(self) -> np.ndarray:
        return self.words()[self.lead:self.lead + self.n]

    def payload_f32(self) -> np.ndarray:
        return self.payload_u32().view(np.float32)

    def guards_intact(self) -> bool:
        w = self.words()
        return bool(np.all(w[:self.lead] == CANARY) and np.all(w[self.lead + self.n:] == CANARY))


def bits(x) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)


def same_f32(got, want) -> bool:
    """Bitwise equality, with every NaN equal to every NaN (payloads may differ
    between the GPU and the host CPU)."""
    got = np.asarray(got, dtype=np.float32)
    want = np.asarray(want, dtype=np.float32)
    gn, wn = np.isnan(got), np.isnan(want)
    if not np.array_equal(gn, wn):
        return False
    return np.array_equal(bits(got[~gn]), bits(want[~wn]))
