"""CPU oracle for the packed NR-MMDiT block forward and its rectified-flow epilogues.

TEST INFRASTRUCTURE ONLY.  Plain, slow, obviously correct NumPy code in float64 (integers for
the packer), written from the method's description on the Mage-Flow pages:

* "Mage-Flow: An Efficient Native-Resolution Foundation Model for Image Generation and
  Editing" - PaperReading review (obsidian blog), sections 2.2(2) native-resolution NR-MMDiT,
  2.2(3) packed CFG and operator fusion, 2.2(4) the Diffusion-NFT objective, and 5 (concepts:
  rectified flow, MMDiT, native resolution packing, CFG);
* the hyper.ai summary of the same paper, sections 方法 (method) and 实验 (experiments).

It works one sample at a time with no packing inside the math, so that the packed GPU result
can be checked against per-sample results.  Only the tests, the package's smoke check and the
bench's CPU-baseline leg may import it; the product path never does.  It shares no code with
the CUDA library and does not import it.

Modules: `pack` (first-fit packing and the plan's index buffers), `model` (the block, the
stack ends and the rectified-flow epilogues, with the QK-RMSNorm and fp8 variants), `brute`
(pure-Python loops for the brute-force pins), `fp8` (E4M3 rounding, per-row quantisation and
the quantised linear layer), `grad` (float64 PyTorch restatement of the block and its
reverse-mode gradients, for the block backward).

Parity status: the packer, RoPE, attention, LayerNorm, GELU, the timestep embedding, the
timestep condition (the two-layer SiLU MLP on it: a hand-worked value and planted mistakes), the
stack's composition (embed -> blocks -> final layer) and the CFG sampler's step sum, the
block's residual structure, the interpolation, the loss, the Diffusion-NFT loss, the Euler
step, CFG, the QK-RMSNorm, E4M3 rounding and the block's gradients are each pinned by tests
against closed forms, invariants, brute force, finite differences or hand-computed values.  The
whole-model numbers (a full block with random weights) have no printed worked example on the
pages: "parity unpinned" for the composed block beyond those structural pins.
"""
from . import pack, model, brute, fp8  # noqa: F401
