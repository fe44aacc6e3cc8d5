"""CPU oracle for the QLoRA NF4 hot path -- TEST INFRASTRUCTURE ONLY.

This package is the slow, plain, float64 reference that the CUDA library is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it.
The product path (``bit_nf4_quantized_39_b300``) never imports, links or
executes anything here, and this package imports nothing from the product.
The two share no code, tables or constants: the oracle builds its own NF4
codebook from the normal-quantile construction, while the CUDA side carries
its own literal table.

Modules
-------
``nf4``     codebook, block absmax, nearest-level search, nibble packing,
            double quantisation of the absmax constants, dequantisation.
``exact``   exact rational helpers (exact mean of fp32 values, correct
            rounding of a rational to fp32 / bf16).
``layer``   the QLoRA linear layer forward ``Y``, backward ``dX`` and the
            adapter gradients ``dA``, ``dB`` in float64.
``loftq``   the LoftQ alternation with an exact LAPACK SVD, and its one-step
            variant that keeps a given quantised weight.
``merge``   merge / unmerge of an adapter into an NF4 weight (dequantise,
            add or subtract s B A, requantise).

Sources (pages of the method, cited by title and section)
--------------------------------------------------------
* "QLoRA technical analysis" (xdnf.cn/news/354788) §2.1: per-tensor absmax
  normalisation followed by a per-element nearest-codebook search (argmin).
* "QLoRA paper summary" (blog.csdn.net, QLoRA论文概述): NF4 is built from
  normal quantiles; double quantisation re-quantises the quantisation
  constants; gradients flow through the frozen 4-bit weight into LoRA.
* "PEFT course notes" (demo.tomabc.com, 高效微调方法) §2.2 / §2.5: W in R^{d x k},
  B in R^{d x r}, A in R^{r x k}, h = Wx + BAx, (d+k) r trainable parameters;
  §4.2: NF4 + double quantisation.
* "PEFT quantization guide" (huggingface docs, 量化): bf16 compute dtype,
  nested (double) quantisation, dequantise-add-requantise merge semantics,
  one-step LoftQ (replace_lora_weights_loftq) that only refits the adapter.
* "LoftQ explainer" (mhpn.cn/news/832204) §2.2 objective
  min ||W - (Q + Delta)||_F^2 with rank(Delta) <= r, §2.3 alternation
  (round-to-nearest Q-step, truncated-SVD Delta-step).

Pins (tests that tie each function to something other than itself) live in
``tests/test_oracle_*.py``.  Every oracle function is pinned; none is
"parity unpinned".
"""

from . import exact, nf4, layer, loftq, merge  # noqa: F401
