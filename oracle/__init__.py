"""CPU oracle for the int4g path -- test infrastructure only (see int4g_oracle)."""
