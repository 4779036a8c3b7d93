"""Oracle for native-resolution packing (first-fit under a fixed token budget) and the index
buffers that describe a pack.

The pages (PaperReading review §2.2(2); hyper.ai summary, 方法) say that images of any size
are flattened to variable-length latent-token sequences and, together with variable-length
text, concatenated by cumulative offsets into one batch under a fixed token budget, with
attention restricted to each sample and each sample keeping its own positions.  The packing
rule itself is not given; the reading taken here is first-fit in candidate order: take
candidate i iff it still fits the remaining budget, otherwise skip it and go on.

Layout conventions (shared with the C library by specification, not by code):
* joint order of a sample: [text tokens | frame 0 (row-major) | frame 1 (row-major)];
* stream order: all text tokens of the packed samples in pack order ("txt" stream), and all
  image tokens in pack order ("img" stream);
* pos[j] = (frame, row, col) of joint token j; text tokens sit at (0, 0, 0).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


class PackError(ValueError):
    def __init__(self, code: str, msg: str):
        super().__init__(f"{code}: {msg}")
        self.code = code


@dataclass
class Plan:
    order: np.ndarray        # [S]   candidate index of each packed sequence
    cu_seqlens: np.ndarray   # [S+1] joint-token offsets
    cu_txt: np.ndarray       # [S+1] text-stream row offsets
    cu_img: np.ndarray       # [S+1] image-stream row offsets
    pos: np.ndarray          # [N][3] (frame, row, col) per joint token
    txt_seq: np.ndarray      # [N_t] sequence of each text row
    txt_joint: np.ndarray    # [N_t] joint token of each text row
    img_seq: np.ndarray      # [N_i] sequence of each image row
    img_joint: np.ndarray    # [N_i] joint token of each image row
    img_pair: np.ndarray     # [N_i] CFG partner image row, -1 if none
    img_target: np.ndarray   # [N_i] 1 if the row belongs to the target (noised, supervised) frame

    @property
    def n_seq(self) -> int:
        return len(self.order)

    @property
    def n_tok(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def n_txt(self) -> int:
        return int(self.cu_txt[-1])

    @property
    def n_img(self) -> int:
        return int(self.cu_img[-1])


def sample_length(s) -> int:
    return s.txt_len + s.frames * s.lat_h * s.lat_w


def validate(samples, budget: int) -> None:
    if budget < 1:
        raise PackError("budget", f"budget {budget} < 1")
    for i, s in enumerate(samples):
        if s.txt_len < 0 or s.lat_h < 1 or s.lat_w < 1 or s.frames not in (1, 2):
            raise PackError("invalid_arg", f"sample {i} has a bad shape")
        if s.cfg_role not in (0, 1, 2):
            raise PackError("invalid_arg", f"sample {i} has cfg_role {s.cfg_role}")
        if sample_length(s) > budget:
            raise PackError("sample_too_long", f"sample {i} ({sample_length(s)} tokens) > {budget}")


def first_fit(samples, budget: int) -> list[int]:
    """Candidate indices taken by first-fit with skip, in candidate order."""
    validate(samples, budget)
    used, taken = 0, []
    for i, s in enumerate(samples):
        length = sample_length(s)
        if used + length <= budget:
            taken.append(i)
            used += length
    return taken


def build_plan(samples, budget: int) -> Plan:
    order = first_fit(samples, budget)
    seq_of_cand = {c: k for k, c in enumerate(order)}
    S = len(order)
    cu, cut, cui = [0], [0], [0]
    for c in order:
        s = samples[c]
        cu.append(cu[-1] + sample_length(s))
        cut.append(cut[-1] + s.txt_len)
        cui.append(cui[-1] + s.frames * s.lat_h * s.lat_w)
    N, Nt, Ni = cu[-1], cut[-1], cui[-1]
    pos = np.zeros((N, 3), dtype=np.int32)
    txt_seq = np.zeros(Nt, np.int32)
    txt_joint = np.zeros(Nt, np.int32)
    img_seq = np.zeros(Ni, np.int32)
    img_joint = np.zeros(Ni, np.int32)
    img_pair = np.full(Ni, -1, np.int32)
    img_target = np.zeros(Ni, np.int32)
    for k, c in enumerate(order):
        s = samples[c]
        j = cu[k]
        for a in range(s.txt_len):
            r = cut[k] + a
            txt_seq[r] = k
            txt_joint[r] = j + a
        j += s.txt_len
        local = 0
        for f in range(s.frames):
            for row in range(s.lat_h):
                for col in range(s.lat_w):
                    r = cui[k] + local
                    img_seq[r] = k
                    img_joint[r] = j + local
                    pos[j + local] = (f, row, col)
                    img_target[r] = 1 if f == s.frames - 1 else 0
                    local += 1
        if s.cfg_role != 0:
            p = s.cfg_pair
            if p not in seq_of_cand:
                raise PackError("invalid_arg", f"CFG partner {p} of candidate {c} is not packed")
            q = samples[p]
            want = 2 if s.cfg_role == 1 else 1
            if (q.cfg_role != want or q.cfg_pair != c or q.frames != s.frames
                    or q.lat_h != s.lat_h or q.lat_w != s.lat_w):
                raise PackError("invalid_arg", f"CFG pair ({c}, {p}) does not match")
            kp = seq_of_cand[p]
            for local in range(s.frames * s.lat_h * s.lat_w):
                img_pair[cui[k] + local] = cui[kp] + local
    a32 = lambda v: np.asarray(v, dtype=np.int32)                    # noqa: E731
    return Plan(a32(order), a32(cu), a32(cut), a32(cui), pos, txt_seq, txt_joint, img_seq,
                img_joint, img_pair, img_target)
