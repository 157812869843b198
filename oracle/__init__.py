"""fp64 CPU oracle (test infrastructure only; see rnn_oracle)."""
