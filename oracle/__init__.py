"""fp64 CPU oracle for the noisy top-k MoE forward pass (test infrastructure;
see ``oracle.moe_oracle``).  Never imported by the library's CUDA path."""
